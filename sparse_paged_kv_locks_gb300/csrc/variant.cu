// Scoring from rank / precision variant records (LOCKS reading notes §4.2
// Eq.(4) with the §6 ablation's ranks and basis precisions):
//   s_hat_j(q_g) = ln sum_{i<16} exp((q_g . mu_j + (V_j^T q_g) . c_i) / sqrt(d))
// from a variant record (include/locks.h): basis codes [128][r] d-major,
// bit-packed little-endian with `vbits` bits, int8 C [16][r], int8 mu,
// fp16 scales.  This is the ablation's path, not the shipped hot path: the
// record is decoded to fp32 in shared memory and the products run on CUDA
// cores.  One CTA per 16 pages of one (sequence, KV head), a warp per page.
#include "common.cuh"
#include "launch.h"

namespace locks {

constexpr int kVarWarps = 4;
constexpr int kVarPagesPerCta = 16;
constexpr int kVarMaxRank = 15;

struct VarWarpSmem {
  float V[kDim][kVarMaxRank + 1];
  float C[kPage][kVarMaxRank + 1];
  float mu[kDim];
  float proj[kMaxGroup][kVarMaxRank + 2];  // [g][k], k = r holds q . mu
};

__host__ __device__ __forceinline__ int var_payload(int r, int vbits) {
  return 16 * r * vbits + 16 * r + kDim + 2 * r + 2 * kPage + 2;
}
__host__ __device__ __forceinline__ int var_stride(int r, int vbits) {
  return (var_payload(r, vbits) + 15) / 16 * 16;
}

__global__ void __launch_bounds__(32 * kVarWarps)
    score_variant_kernel(const __nv_bfloat16 *__restrict__ q,
                         const uint8_t *__restrict__ records, int r, int vbits,
                         const int32_t *__restrict__ seq_lens, int h_kv,
                         int G, int max_pages, float *__restrict__ scores,
                         int32_t *status) {
  extern __shared__ __align__(16) uint8_t smem[];
  float *sq = reinterpret_cast<float *>(smem);  // [G][128]
  VarWarpSmem *ws_all =
      reinterpret_cast<VarWarpSmem *>(smem + sizeof(float) * kMaxGroup * kDim);
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int b = blockIdx.z, h = blockIdx.y;
  VarWarpSmem &ws = ws_all[wid];
  int L = seq_lens[b];
  if (L < 0 || L > max_pages * kPage) {
    if (threadIdx.x == 0 && h == 0 && blockIdx.x == 0)
      set_status(status, LOCKS_DEV_BAD_SEQ_LEN);
    L = max(0, min(L, max_pages * kPage));
  }
  const int nf = L / kPage;
  const int j0 = blockIdx.x * kVarPagesPerCta;
  if (j0 >= nf) return;
  const __nv_bfloat16 *qb = q + ((size_t)b * h_kv + h) * G * kDim;
  for (int e = threadIdx.x; e < G * kDim; e += blockDim.x)
    sq[e] = __bfloat162float(qb[e]);
  __syncthreads();

  const size_t stride = (size_t)var_stride(r, vbits);
  const int off_c = 16 * r * vbits, off_mu = off_c + 16 * r;
  const int off_sv = off_mu + kDim, off_sc = off_sv + 2 * r;
  const int off_smu = off_sc + 2 * kPage;
  const uint32_t cmask = (1u << vbits) - 1u, sbit = 1u << (vbits - 1);
  const float rsd = 0.08838834764831845f;  // 1/sqrt(128)
  for (int j = j0 + wid; j < min(nf, j0 + kVarPagesPerCta); j += kVarWarps) {
    const uint8_t *rec =
        records + (((size_t)b * h_kv + h) * max_pages + j) * stride;
    // basis: this lane's 4 dims x r codes start at byte lane * r * vbits / 2
    const uint8_t *vb = rec + lane * r * vbits / 2;
    for (int idx = 0; idx < 4 * r; ++idx) {
      const int bit = idx * vbits;
      uint32_t c = ((uint32_t)vb[bit >> 3] >> (bit & 7)) & cmask;
      const int code = (c & sbit) ? (int)c - (int)(cmask + 1) : (int)c;
      const int dj = idx / r, k = idx - dj * r;
      const float sv = __half2float(
          *reinterpret_cast<const __half *>(rec + off_sv + 2 * k));
      ws.V[4 * lane + dj][k] = (float)code * sv;
    }
    for (int e = lane; e < kPage * r; e += 32) {
      const int i = e / r, k = e - i * r;
      const float sc = __half2float(
          *reinterpret_cast<const __half *>(rec + off_sc + 2 * i));
      ws.C[i][k] = (float)(int8_t)rec[off_c + e] * sc;
    }
    const float smu =
        __half2float(*reinterpret_cast<const __half *>(rec + off_smu));
#pragma unroll
    for (int dj = 0; dj < 4; ++dj)
      ws.mu[4 * lane + dj] = (float)(int8_t)rec[off_mu + 4 * lane + dj] * smu;
    __syncwarp();
    // projections V^T q_g (k < r) and q_g . mu (k = r)
    for (int t = lane; t < G * (r + 1); t += 32) {
      const int g = t / (r + 1), k = t - g * (r + 1);
      const float *qg = sq + g * kDim;
      float acc = 0.f;
      if (k < r) {
        for (int d = 0; d < kDim; ++d) acc = fmaf(ws.V[d][k], qg[d], acc);
      } else {
        for (int d = 0; d < kDim; ++d) acc = fmaf(ws.mu[d], qg[d], acc);
      }
      ws.proj[g][k] = acc;
    }
    __syncwarp();
    // logits of (g, token i) in 16-lane groups, then the 16-token LSE
    for (int base = 0; base < G * kPage; base += 32) {
      const int t = base + lane, g = t / kPage, i = t - g * kPage;
      float x = -INFINITY;
      if (g < G) {
        float acc = ws.proj[g][r];
        for (int k = 0; k < r; ++k) acc = fmaf(ws.proj[g][k], ws.C[i][k], acc);
        x = acc * rsd;
      }
      float m = x;
#pragma unroll
      for (int o = 1; o < 16; o <<= 1)
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      float e = g < G ? expf(x - m) : 0.f;
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) e += __shfl_xor_sync(0xffffffffu, e, o);
      if (g < G && i == 0)
        scores[(((size_t)b * h_kv + h) * G + g) * max_pages + j] =
            m + logf(e);
    }
    __syncwarp();
  }
}

size_t variant_record_bytes(int rank, int vbits) {
  return (size_t)var_stride(rank, vbits);
}

cudaError_t launch_score_variant(const void *q, const void *records,
                                 int rank, int vbits,
                                 const int32_t *seq_lens, int batch, int h_kv,
                                 int G, int max_pages, float *scores,
                                 int32_t *status, cudaStream_t stream) {
  const size_t smem = sizeof(float) * kMaxGroup * kDim +
                      sizeof(VarWarpSmem) * kVarWarps;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(
        score_variant_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
        (int)smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid((max_pages + kVarPagesPerCta - 1) / kVarPagesPerCta, h_kv, batch);
  score_variant_kernel<<<grid, 32 * kVarWarps, smem, stream>>>(
      static_cast<const __nv_bfloat16 *>(q),
      static_cast<const uint8_t *>(records), rank, vbits, seq_lens, h_kv, G,
      max_pages, scores, status);
  return cudaGetLastError();
}

}  // namespace locks
