// Scoring from rank / precision variant records (LOCKS reading notes §4.2
// Eq.(4) with the §6 ablation's ranks and basis precisions):
//   s_hat_j(q_g) = ln sum_{i<16} exp((q_g . mu_j + (V_j^T q_g) . c_i) / sqrt(d))
// from a variant record (include/locks.h): basis codes [128][r] d-major,
// bit-packed little-endian with `vbits` bits, int8 C [16][r], int8 mu,
// fp16 scales, 16 B stride.  This is the ablation's path, not the shipped
// tensor-core path; it runs on CUDA cores for every (r, vbits).
//
// A warp per record: the record is staged in shared memory with 16-byte
// loads; lane l decodes the codes of head dims 4l..4l+3 (4 r codes, which
// never straddle a 32-bit word since vbits divides 32) into registers with
// shifts fixed at compile time (one instantiation per (r, vbits)); for
// each query head the r + 1 partial products (V^T q and q . mu) over the
// lane's dims are reduced across the warp with a 16-value reduce-scatter;
// the 16 x G logits then take one (token, head) pair per lane and the
// 16-token log-sum-exp runs in groups of 16 lanes.
#include "common.cuh"
#include "launch.h"

namespace locks {

constexpr int kVarWarps = 8;
constexpr int kVarPagesPerWarp = 8;
constexpr int kVarPagesPerCta = kVarWarps * kVarPagesPerWarp;
constexpr int kVarMaxRank = 15;
constexpr int kVarMaxStride = 2368;  // largest record stride (r 15, 8 bits)

__host__ __device__ __forceinline__ int var_payload(int r, int vbits) {
  return 16 * r * vbits + 16 * r + kDim + 2 * r + 2 * kPage + 2;
}
__host__ __device__ __forceinline__ int var_stride(int r, int vbits) {
  return (var_payload(r, vbits) + 15) / 16 * 16;
}

struct alignas(16) VarWarpSmem {
  uint8_t rec[kVarMaxStride];        // the staged record
  float proj[kMaxGroup][16];         // [g][k]: sV_k (V_k^T q_g); k = r: q.mu
  float cf[kPage][kVarMaxRank + 2];  // sC_i C[i][k] (rows padded: 17)
};

// 16-value reduce-scatter: lane l ends with the warp sum of v[l % 16].
__device__ __forceinline__ float var_reduce16(float (&v)[16], int lane) {
#pragma unroll
  for (int o = 8; o >= 1; o >>= 1) {
    const bool hi = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      const float send = hi ? v[i] : v[i + o];
      const float keep = hi ? v[i + o] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 16);
}

template <int R, int VB>
__global__ void __launch_bounds__(32 * kVarWarps)
    score_variant_kernel(const __nv_bfloat16 *__restrict__ q,
                         const uint8_t *__restrict__ records,
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

  constexpr int stride = (16 * R * VB + 16 * R + kDim + 2 * R + 2 * kPage +
                          2 + 15) / 16 * 16;
  constexpr int off_c = 16 * R * VB, off_mu = off_c + 16 * R;
  constexpr int off_sv = off_mu + kDim, off_sc = off_sv + 2 * R;
  constexpr int off_smu = off_sc + 2 * kPage;
  constexpr uint32_t cmask = (1u << VB) - 1u, sbit = 1u << (VB - 1);
  // 32-bit words that cover one lane's 4 R VB code bits (plus one for a
  // start that is not word-aligned)
  constexpr int kLaneWords = (4 * R * VB + 31) / 32;
  const float rsd = 0.08838834764831845f;  // 1/sqrt(128)
  const uint32_t *rw = reinterpret_cast<const uint32_t *>(ws.rec);

  for (int j = j0 + wid; j < min(nf, j0 + kVarPagesPerCta); j += kVarWarps) {
    const uint4 *src = reinterpret_cast<const uint4 *>(
        records + (((size_t)b * h_kv + h) * max_pages + j) * (size_t)stride);
    for (int c = lane; c < stride / 16; c += 32)
      reinterpret_cast<uint4 *>(ws.rec)[c] = __ldg(src + c);
    __syncwarp();
    // this lane's codes: dims 4l + dj, component k at bit
    // 4 l R VB + (dj R + k) VB; the lane's 4 R VB bits start at bit
    // 4 l R VB, which is word-aligned when 4 R VB is a multiple of 32 and
    // otherwise read from the words that cover it
    float code[4][R];
    {
      const int bit0 = 4 * lane * R * VB;
      const int w0 = bit0 >> 5, sh0 = bit0 & 31;
      uint32_t wv[kLaneWords + 1];
#pragma unroll
      for (int i = 0; i <= kLaneWords; ++i)
        wv[i] = (w0 + i) * 4 < stride ? rw[w0 + i] : 0u;
      // realign so the lane's first code sits at bit 0 of wv[0]; every
      // later shift is then a compile-time constant
      if ((4 * R * VB) % 32 != 0) {
#pragma unroll
        for (int i = 0; i < kLaneWords; ++i)
          wv[i] = __funnelshift_r(wv[i], wv[i + 1], sh0);
      }
#pragma unroll
      for (int idx = 0; idx < 4 * R; ++idx) {
        const int bit = idx * VB;  // codes never straddle a word
        const uint32_t u = (wv[bit >> 5] >> (bit & 31)) & cmask;
        code[idx / R][idx % R] =
            (float)((u & sbit) ? (int)u - (int)(cmask + 1) : (int)u);
      }
    }
    float mu[4];
#pragma unroll
    for (int dj = 0; dj < 4; ++dj)
      mu[dj] = (float)(int8_t)ws.rec[off_mu + 4 * lane + dj];
    const float smu =
        __half2float(*reinterpret_cast<const __half *>(ws.rec + off_smu));
    const int kk = lane & 15;  // component this lane keeps after a reduction
    const float sv_k = kk < R ? __half2float(*reinterpret_cast<const __half *>(
                                    ws.rec + off_sv + 2 * kk))
                              : 0.f;
    // projections, one head at a time
#pragma unroll 1
    for (int g = 0; g < G; ++g) {
      const float4 qv = reinterpret_cast<const float4 *>(sq + g * kDim)[lane];
      const float qd[4] = {qv.x, qv.y, qv.z, qv.w};
      float v[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) v[k] = 0.f;
#pragma unroll
      for (int k = 0; k < R; ++k)
#pragma unroll
        for (int dj = 0; dj < 4; ++dj) v[k] = fmaf(code[dj][k], qd[dj], v[k]);
#pragma unroll
      for (int dj = 0; dj < 4; ++dj) v[R] = fmaf(mu[dj], qd[dj], v[R]);
      const float t = var_reduce16(v, lane);
      if (lane < 16 && kk <= R)
        ws.proj[g][kk] = kk < R ? t * sv_k : t * smu;
    }
    // coefficients, dequantised
    for (int e = lane; e < kPage * R; e += 32) {
      const int i = e / R, k = e - i * R;
      const float sc =
          __half2float(*reinterpret_cast<const __half *>(ws.rec + off_sc + 2 * i));
      ws.cf[i][k] = (float)(int8_t)ws.rec[off_c + e] * sc;
    }
    __syncwarp();
    // logits of (head g, token i), 16 lanes per head, then the 16-token LSE
    for (int base = 0; base < G * kPage; base += 32) {
      const int t = base + lane, g = t >> 4, i = t & 15;
      float x = -INFINITY;
      if (g < G) {
        float acc = ws.proj[g][R];
#pragma unroll
        for (int k = 0; k < R; ++k) acc = fmaf(ws.proj[g][k], ws.cf[i][k], acc);
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

template <int R, int VB>
static cudaError_t launch_variant(const void *q, const void *records,
                                  const int32_t *seq_lens, int batch,
                                  int h_kv, int G, int max_pages,
                                  float *scores, int32_t *status,
                                  cudaStream_t stream) {
  const size_t smem =
      sizeof(float) * kMaxGroup * kDim + sizeof(VarWarpSmem) * kVarWarps;
  dim3 grid((max_pages + kVarPagesPerCta - 1) / kVarPagesPerCta, h_kv, batch);
  cudaError_t e = cudaFuncSetAttribute(score_variant_kernel<R, VB>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  score_variant_kernel<R, VB><<<grid, 32 * kVarWarps, smem, stream>>>(
      static_cast<const __nv_bfloat16 *>(q),
      static_cast<const uint8_t *>(records), seq_lens, h_kv, G, max_pages,
      scores, status);
  return cudaGetLastError();
}

template <int R>
static cudaError_t launch_variant_rank(const void *q, const void *records,
                                       int vbits, const int32_t *seq_lens,
                                       int batch, int h_kv, int G,
                                       int max_pages, float *scores,
                                       int32_t *status, cudaStream_t stream) {
  switch (vbits) {
    case 2:
      return launch_variant<R, 2>(q, records, seq_lens, batch, h_kv, G,
                                  max_pages, scores, status, stream);
    case 4:
      return launch_variant<R, 4>(q, records, seq_lens, batch, h_kv, G,
                                  max_pages, scores, status, stream);
    case 8:
      return launch_variant<R, 8>(q, records, seq_lens, batch, h_kv, G,
                                  max_pages, scores, status, stream);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_score_variant(const void *q, const void *records,
                                 int rank, int vbits,
                                 const int32_t *seq_lens, int batch, int h_kv,
                                 int G, int max_pages, float *scores,
                                 int32_t *status, cudaStream_t stream) {
  switch (rank) {
    case 4:
      return launch_variant_rank<4>(q, records, vbits, seq_lens, batch, h_kv,
                                    G, max_pages, scores, status, stream);
    case 8:
      return launch_variant_rank<8>(q, records, vbits, seq_lens, batch, h_kv,
                                    G, max_pages, scores, status, stream);
    case 12:
      return launch_variant_rank<12>(q, records, vbits, seq_lens, batch, h_kv,
                                     G, max_pages, scores, status, stream);
    case 15:
      return launch_variant_rank<15>(q, records, vbits, seq_lens, batch, h_kv,
                                     G, max_pages, scores, status, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace locks
