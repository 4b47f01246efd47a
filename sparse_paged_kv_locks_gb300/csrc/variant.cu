// Scoring from rank / precision variant records (LOCKS reading notes §4.2
// Eq.(4) with the §6 ablation's ranks and basis precisions):
//   s_hat_j(q_g) = ln sum_{i<16} exp((q_g . mu_j + (V_j^T q_g) . c_i) / sqrt(d))
// from a variant record (include/locks.h): basis codes [128][r] d-major,
// bit-packed little-endian with `vbits` bits, int8 C [16][r], int8 mu,
// fp16 scales, 16 B stride.  This is the ablation's path; the shipped
// (8, 4-bit) record has its own layout and scoring kernel.
//
// A warp per record, one instantiation per (r, vbits), records
// double-buffered in shared memory with 16-byte cp.async.  Lane l decodes
// the codes of head dims 4l..4l+3 (4 r codes, which never straddle a 32-bit
// word since vbits divides 32; shifts fixed at compile time) and writes
// them as bf16 into a 16 x 128 operand tile: rows 0..r-1 the basis
// columns, row r the centroid codes, the rest zero.  Eight bf16 mma.sync
// (m16n8k16, K = 128 head dims, N = 8 query heads per tile) give every
// component's V_k^T q_g and q_g . mu at once, exactly up to fp32
// accumulation (the codes and the bf16 query are exact bf16 operands).
// Scaled by sV_k (smu for the centroid row), the projections go to shared
// memory; the 16 x G logits then take one token and two heads per lane in
// fp32 and the 16-token log-sum-exp runs in groups of 16 lanes.
#include "common.cuh"
#include "launch.h"

namespace locks {

constexpr int kVarWarps = 8;
constexpr int kVarPagesPerWarp = 8;
constexpr int kVarPagesPerCta = kVarWarps * kVarPagesPerWarp;
// staged query rows, bf16, padded so the B-fragment loads of the eight
// rows of a tile fall in distinct banks
constexpr int kVarQStride = kDim + 8;
constexpr int kVarQBytes = kMaxGroup * kVarQStride * 2;
// projections [row][head]; even stride so a lane reads two heads at once
constexpr int kVarPStride = kMaxGroup + 2;
constexpr int kVarTileBytes = 16 * kDim * 2;

__host__ __device__ __forceinline__ int var_payload(int r, int vbits) {
  return 16 * r * vbits + 16 * r + kDim + 2 * r + 2 * kPage + 2;
}
__host__ __device__ __forceinline__ int var_stride(int r, int vbits) {
  return (var_payload(r, vbits) + 15) / 16 * 16;
}

template <int R, int VB>
struct VarLayout {
  static constexpr int stride = (16 * R * VB + 16 * R + kDim + 2 * R +
                                 2 * kPage + 2 + 15) / 16 * 16;
  static constexpr int off_c = 16 * R * VB;
  static constexpr int off_mu = off_c + 16 * R;
  static constexpr int off_sv = off_mu + kDim;
  static constexpr int off_sc = off_sv + 2 * R;
  static constexpr int off_smu = off_sc + 2 * kPage;
  // per warp: two staged records, the operand tile, the projections
  static constexpr int warp_bytes =
      2 * stride + kVarTileBytes + 16 * kVarPStride * 4;
  static constexpr int smem_bytes = kVarQBytes + kVarWarps * warp_bytes;
};

// byte offset of head dims 8c..8c+7 of operand row `row` (16-byte chunks
// XOR-swizzled by the row, so ldmatrix's eight rows hit distinct banks)
__device__ __forceinline__ uint32_t var_swz(int row, int c) {
  return (uint32_t)(row * (kDim * 2) + ((c ^ (row & 7)) << 4));
}

__device__ __forceinline__ uint32_t var_pack_bf2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

template <int R, int VB>
__global__ void __launch_bounds__(32 * kVarWarps, 3)
    score_variant_kernel(const __nv_bfloat16 *__restrict__ q,
                         const uint8_t *__restrict__ records,
                         const int32_t *__restrict__ seq_lens, int h_kv,
                         int G, int max_pages, float *__restrict__ scores,
                         int32_t *status) {
  using Ly = VarLayout<R, VB>;
  static_assert(R + 1 <= 16, "basis rows and the centroid row fit 16 rows");
  extern __shared__ __align__(16) uint8_t smem[];
  __nv_bfloat16 *sq = reinterpret_cast<__nv_bfloat16 *>(smem);
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int gq = lane >> 2, t4 = lane & 3;
  const int b = blockIdx.z, h = blockIdx.y;
  uint8_t *wsm = smem + kVarQBytes + (size_t)wid * Ly::warp_bytes;
  uint8_t *stage = wsm;                         // [2][stride]
  uint8_t *tile = wsm + 2 * Ly::stride;         // [16][128] bf16, swizzled
  float *ps = reinterpret_cast<float *>(tile + kVarTileBytes);

  int L = seq_lens[b];
  if (L < 0 || L > max_pages * kPage) {
    if (threadIdx.x == 0 && h == 0 && blockIdx.x == 0)
      set_status(status, LOCKS_DEV_BAD_SEQ_LEN);
    L = max(0, min(L, max_pages * kPage));
  }
  const int nf = L / kPage;
  const int j0 = blockIdx.x * kVarPagesPerCta;
  if (j0 >= nf) return;
  // the group's query rows as bf16 (rows >= G zero)
  const __nv_bfloat16 *qb = q + ((size_t)b * h_kv + h) * G * kDim;
  for (int e = threadIdx.x; e < kMaxGroup * kDim; e += blockDim.x) {
    const int row = e / kDim, d = e - row * kDim;
    sq[row * kVarQStride + d] =
        row < G ? qb[row * kDim + d] : __float2bfloat16(0.f);
  }
  // operand rows below the centroid row stay zero
  for (int c = lane; c < (15 - R) * kDim * 2 / 16; c += 32)
    reinterpret_cast<uint4 *>(tile + (R + 1) * kDim * 2)[c] =
        make_uint4(0u, 0u, 0u, 0u);
  __syncthreads();

  const int jend = min(nf, j0 + kVarPagesPerCta);
  const int first = j0 + wid;
  const int n_my = first < jend ? (jend - first + kVarWarps - 1) / kVarWarps
                                : 0;
  if (n_my == 0) return;
  const uint8_t *src0 =
      records + ((size_t)b * h_kv + h) * max_pages * (size_t)Ly::stride;
  auto issue = [&](int t) {
    const uint8_t *src = src0 + (size_t)(first + t * kVarWarps) * Ly::stride;
    const uint32_t dst = smem_u32(stage + (t & 1) * Ly::stride);
    for (int c = lane; c < Ly::stride / 16; c += 32)
      cp_async16(dst + 16 * c, src + 16 * c);
  };
  constexpr float kLog2eRsqrtD = 0.12751743074602467f;  // log2(e)/sqrt(128)
  constexpr float kLn2 = 0.69314718055994531f;
  constexpr int kLaneWords = (4 * R * VB + 31) / 32;
  const uint32_t tile_s = smem_u32(tile);
  const int ntiles = G > 8 ? 2 : 1;
  const int i_tok = lane & 15;
  float *out = scores + ((size_t)b * h_kv + h) * G * (size_t)max_pages;

  // B fragments of heads 0..7 (dims 16 s + 2 t4 + {0, 1, 8, 9}), kept in
  // registers; heads 8..15 are read from shared memory when G > 8
  uint32_t qf[8][2];
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const __nv_bfloat16 *qr = sq + gq * kVarQStride + 16 * s + 2 * t4;
    qf[s][0] = *reinterpret_cast<const uint32_t *>(qr);
    qf[s][1] = *reinterpret_cast<const uint32_t *>(qr + 8);
  }

  issue(0);
  cp_async_commit();
  for (int t = 0; t < n_my; ++t) {
    if (t + 1 < n_my) issue(t + 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncwarp();
    const uint8_t *rec = stage + (t & 1) * Ly::stride;
    const int j = first + t * kVarWarps;

    // 1. this lane's codes (dims 4l..4l+3, component k at relative bit
    //    (dj R + k) VB) and centroid codes -> operand rows 0..R
    {
      uint32_t wv[kLaneWords + 1];
      if constexpr ((4 * R * VB) % 32 == 0) {
        // kLaneWords whole words from byte 4 kLaneWords l: 16-, 8- or 4-byte
        // loads as the alignment allows
        constexpr int kVec = kLaneWords % 4 == 0 ? 4
                             : kLaneWords % 2 == 0 ? 2 : 1;
        const uint8_t *lw = rec + 4 * kLaneWords * lane;
#pragma unroll
        for (int w = 0; w < kLaneWords; w += kVec) {
          if constexpr (kVec == 4) {
            const uint4 v = *reinterpret_cast<const uint4 *>(lw + 4 * w);
            wv[w] = v.x; wv[w + 1] = v.y; wv[w + 2] = v.z; wv[w + 3] = v.w;
          } else if constexpr (kVec == 2) {
            const uint2 v = *reinterpret_cast<const uint2 *>(lw + 4 * w);
            wv[w] = v.x; wv[w + 1] = v.y;
          } else {
            wv[w] = *reinterpret_cast<const uint32_t *>(lw + 4 * w);
          }
        }
        wv[kLaneWords] = 0u;
      } else {  // the lane's bits start mid-word: realign with funnel shifts
        const uint32_t *rw = reinterpret_cast<const uint32_t *>(rec);
        const int bit0 = 4 * lane * R * VB;
        const int w0 = bit0 >> 5, sh0 = bit0 & 31;
#pragma unroll
        for (int w = 0; w <= kLaneWords; ++w)
          wv[w] = (w0 + w) * 4 < Ly::stride ? rw[w0 + w] : 0u;
#pragma unroll
        for (int w = 0; w < kLaneWords; ++w)
          wv[w] = __funnelshift_r(wv[w], wv[w + 1], sh0);
      }
      const uint32_t part = (uint32_t)(lane & 1) * 8;
#pragma unroll
      for (int k = 0; k < R; ++k) {
        float f[4];
#pragma unroll
        for (int dj = 0; dj < 4; ++dj) {
          const int bit = (dj * R + k) * VB;
          f[dj] = (float)((int32_t)(wv[bit >> 5] << (32 - VB - (bit & 31))) >>
                          (32 - VB));
        }
        *reinterpret_cast<uint2 *>(tile + var_swz(k, lane >> 1) + part) =
            make_uint2(var_pack_bf2(f[0], f[1]), var_pack_bf2(f[2], f[3]));
      }
      const uint32_t mw =
          *reinterpret_cast<const uint32_t *>(rec + Ly::off_mu + 4 * lane);
      *reinterpret_cast<uint2 *>(tile + var_swz(R, lane >> 1) + part) =
          make_uint2(var_pack_bf2((float)(int8_t)(mw & 0xff),
                                  (float)(int8_t)((mw >> 8) & 0xff)),
                     var_pack_bf2((float)(int8_t)((mw >> 16) & 0xff),
                                  (float)(int8_t)(mw >> 24)));
    }
    // this lane's token row of coefficient codes and its scale
    float cr[R];
    if constexpr (R % 4 == 0) {
      const uint32_t *cw =
          reinterpret_cast<const uint32_t *>(rec + Ly::off_c + i_tok * R);
#pragma unroll
      for (int w = 0; w < R / 4; ++w) {
        const uint32_t x = cw[w];
#pragma unroll
        for (int u = 0; u < 4; ++u)
          cr[4 * w + u] = (float)(int8_t)((x >> (8 * u)) & 0xff);
      }
    } else {
#pragma unroll
      for (int k = 0; k < R; ++k)
        cr[k] = (float)(int8_t)rec[Ly::off_c + i_tok * R + k];
    }
    const float sci = __half2float(
        *reinterpret_cast<const __half *>(rec + Ly::off_sc + 2 * i_tok));
    __syncwarp();

    // 2. D[row][head] = sum_d tile[row][d] q[head][d] on tensor cores
    float d[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    {
      const int mi = lane >> 3, arow = (lane & 7) + 8 * (mi & 1);
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        uint32_t a[4];
        if constexpr (R + 1 <= 8) {  // rows 8..15 are zero: two matrices
          uint32_t a2[2];
          ldmatrix_x2(a2, tile_s + var_swz(lane & 7, 2 * s + ((lane >> 3) & 1)));
          a[0] = a2[0];
          a[1] = 0u;
          a[2] = a2[1];
          a[3] = 0u;
        } else {
          ldmatrix_x4(a, tile_s + var_swz(arow, 2 * s + (mi >> 1)));
        }
        mma_bf16(d[0], a, qf[s][0], qf[s][1]);
        if (ntiles == 2) {
          const __nv_bfloat16 *qr8 =
              sq + (8 + gq) * kVarQStride + 16 * s + 2 * t4;
          mma_bf16(d[1], a, *reinterpret_cast<const uint32_t *>(qr8),
                   *reinterpret_cast<const uint32_t *>(qr8 + 8));
        }
      }
    }
    // scaled projections: row k < R by sV_k, row R (centroid) by smu
    {
      const int r0 = gq, r1 = gq + 8;
      const float s0 =
          r0 <= R ? __half2float(*reinterpret_cast<const __half *>(
                        rec + (r0 < R ? Ly::off_sv + 2 * r0 : Ly::off_smu)))
                  : 0.f;
      const float s1 =
          r1 <= R ? __half2float(*reinterpret_cast<const __half *>(
                        rec + (r1 < R ? Ly::off_sv + 2 * r1 : Ly::off_smu)))
                  : 0.f;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        if (nt >= ntiles) break;
        const int c = 8 * nt + 2 * t4;
        if (r0 <= R)
          *reinterpret_cast<float2 *>(ps + r0 * kVarPStride + c) =
              make_float2(d[nt][0] * s0, d[nt][1] * s0);
        if (r1 <= R)
          *reinterpret_cast<float2 *>(ps + r1 * kVarPStride + c) =
              make_float2(d[nt][2] * s1, d[nt][3] * s1);
      }
    }
    __syncwarp();

    // 3. logits (log2 units) of token i_tok for heads g, g + 1, then the
    //    LSE over the 16 tokens of each 16-lane half (heads at or above G
    //    have zero projections: finite, not written)
    for (int g0 = 0; g0 < G; g0 += 4) {
      const int g = g0 + 2 * (lane >> 4);
      float a0 = 0.f, a1 = 0.f;
#pragma unroll
      for (int k = 0; k < R; ++k) {
        const float2 pk =
            *reinterpret_cast<const float2 *>(ps + k * kVarPStride + g);
        a0 = fmaf(pk.x, cr[k], a0);
        a1 = fmaf(pk.y, cr[k], a1);
      }
      const float2 pm =
          *reinterpret_cast<const float2 *>(ps + R * kVarPStride + g);
      const float x0 = fmaf(a0, sci, pm.x) * kLog2eRsqrtD;
      const float x1 = fmaf(a1, sci, pm.y) * kLog2eRsqrtD;
      float m0 = x0, m1 = x1;
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) {
        m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, o));
        m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, o));
      }
      float e0 = ex2_fast(x0 - m0), e1 = ex2_fast(x1 - m1);
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) {
        e0 += __shfl_xor_sync(0xffffffffu, e0, o);
        e1 += __shfl_xor_sync(0xffffffffu, e1, o);
      }
      if (i_tok == 0) {
        if (g < G) out[(size_t)g * max_pages + j] = (m0 + lg2_fast(e0)) * kLn2;
        if (g + 1 < G)
          out[(size_t)(g + 1) * max_pages + j] = (m1 + lg2_fast(e1)) * kLn2;
      }
    }
    __syncwarp();  // the stage, the tile and the projections are reused
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
  const size_t smem = VarLayout<R, VB>::smem_bytes;
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
