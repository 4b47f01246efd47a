// Attention over the selected pages (LOCKS reading notes §2 and §4.4
// Algorithm 2: fetch full K/V only for the selected pages, then standard
// softmax attention for every query head of the group).
//
// Split-K flash decode.  A CTA owns one (sequence, KV head, split) and a
// slice of that pair's selected-page list; its four warps take every fourth
// page.  Each warp gathers its pages (one 4 KB K run and one 4 KB V run per
// page through the page table) with 16-byte cp.async into a private, double
// buffered, XOR-swizzled shared-memory tile, so every K/V byte is read once
// for the whole GQA group.  Q K^T and P V run on bf16 mma.sync with the
// query heads as the M dimension; softmax is online in base 2.  Warps merge
// in shared memory; splits merge in a second small kernel.
#include "common.cuh"
#include "launch.h"

namespace locks {

constexpr int kDecWarps = 4;
constexpr int kDecThreads = 32 * kDecWarps;
constexpr int kKvTile = kPage * kDim * 2;                     // 4096 bytes
constexpr int kDecSmem = kDecWarps * 2 * 2 * kKvTile;         // 64 KB
constexpr float kDecScale = 0.12751743074602467f;             // log2e/sqrt(d)
constexpr float kLn2f = 0.69314718055994531f;

__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

// swizzled byte offset of 16-byte chunk `ch` (0..15) of token row `row`
__device__ __forceinline__ uint32_t swz(int row, int ch) {
  return (uint32_t)(row * 256 + ((ch ^ (row & 7)) << 4));
}

template <bool WIDE>
__global__ void __launch_bounds__(kDecThreads)
    decode_kernel(const __nv_bfloat16 *__restrict__ q,
                  const __nv_bfloat16 *__restrict__ k_cache,
                  const __nv_bfloat16 *__restrict__ v_cache, int64_t num_phys,
                  const int32_t *__restrict__ pt,
                  const int32_t *__restrict__ seq_lens,
                  const int32_t *__restrict__ idx, int k, int h_kv, int G,
                  int max_pages, int pps, int n_split,
                  __nv_bfloat16 *__restrict__ o_out,
                  float *__restrict__ lse_out, float *__restrict__ o_part,
                  float *__restrict__ lse_part, int32_t *status) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int gq = lane >> 2, t4 = lane & 3;
  const int h_q = h_kv * G;

  int L = seq_lens[b];
  if (L < 0 || L > max_pages * kPage) {
    if (threadIdx.x == 0 && h == 0 && split == 0)
      set_status(status, LOCKS_DEV_BAD_SEQ_LEN);
    L = max(0, min(L, max_pages * kPage));
  }
  const int n = (L + kPage - 1) / kPage;
  const int list_len = idx ? k : n;
  const int begin = split * pps, end = min(list_len, begin + pps);
  const int32_t *my_idx = idx ? idx + ((size_t)b * h_kv + h) * k : nullptr;
  const int32_t *my_pt = pt + (size_t)b * max_pages;

  // query A fragments (bf16), rows = heads of the group
  uint32_t qa[8][4];
  {
    const __nv_bfloat16 *qb = q + ((size_t)b * h_q + (size_t)h * G) * kDim;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      const int d0 = 16 * s + 2 * t4;
      qa[s][0] = gq < G ? __ldg(reinterpret_cast<const uint32_t *>(qb + gq * kDim + d0)) : 0u;
      qa[s][2] = gq < G ? __ldg(reinterpret_cast<const uint32_t *>(qb + gq * kDim + d0 + 8)) : 0u;
      qa[s][1] = (WIDE && gq + 8 < G) ? __ldg(reinterpret_cast<const uint32_t *>(qb + (gq + 8) * kDim + d0)) : 0u;
      qa[s][3] = (WIDE && gq + 8 < G) ? __ldg(reinterpret_cast<const uint32_t *>(qb + (gq + 8) * kDim + d0 + 8)) : 0u;
    }
  }

  uint8_t *wbase = smem + wid * (4 * kKvTile);  // [stage][K|V]
  const uint32_t wbase_s = smem_u32(wbase);
  // resolve the whole slice (index -> page table -> physical page) at once,
  // so the per-page loop below only issues copies
  int *s_phys = reinterpret_cast<int *>(smem + kDecSmem);
  int *s_ntok = s_phys + pps;
  for (int i = threadIdx.x; i < end - begin; i += blockDim.x) {
    const int pg = my_idx ? my_idx[begin + i] : begin + i;
    int ph = -1, nt = 0;
    if (pg >= n) {
      set_status(status, LOCKS_DEV_BAD_INDEX);
    } else if (pg >= 0) {
      ph = my_pt[pg];
      if (ph < 0 || ph >= num_phys) {
        set_status(status, LOCKS_DEV_BAD_PAGE_ID);
        ph = -1;
      } else {
        nt = min(kPage, L - pg * kPage);
      }
    }
    s_phys[i] = ph;
    s_ntok[i] = nt;
  }
  __syncthreads();
  int e_next = wid;
  // next valid page of this warp's share of the slice
  auto fetch_next = [&](int &phys, int &ntok) -> bool {
    while (e_next < end - begin) {
      const int e = e_next;
      e_next += kDecWarps;
      if (s_phys[e] < 0) continue;
      phys = s_phys[e];
      ntok = s_ntok[e];
      return true;
    }
    return false;
  };
  auto issue = [&](int stage, int phys) {
    const uint8_t *ks = reinterpret_cast<const uint8_t *>(k_cache) +
                        ((size_t)phys * h_kv + h) * kKvTile;
    const uint8_t *vs = reinterpret_cast<const uint8_t *>(v_cache) +
                        ((size_t)phys * h_kv + h) * kKvTile;
    const uint32_t kd = wbase_s + stage * 2 * kKvTile, vd = kd + kKvTile;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int c = lane + 32 * i, row = c >> 4, ch = c & 15;
      cp_async16(kd + swz(row, ch), ks + 16 * c);
      cp_async16(vd + swz(row, ch), vs + 16 * c);
    }
  };

  float o[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_run = -INFINITY, m_run8 = -INFINITY, l_run = 0.f, l_run8 = 0.f;

  int ph0 = 0, nt0 = 0, ph1 = 0, nt1 = 0;
  bool have0 = fetch_next(ph0, nt0);
  if (have0) issue(0, ph0);
  cp_async_commit();
  bool have1 = fetch_next(ph1, nt1);
  if (have1) issue(1, ph1);
  cp_async_commit();

  for (int it = 0;; ++it) {
    const int st = it & 1;
    const bool have = st ? have1 : have0;
    if (!have) break;
    const int ntok = st ? nt1 : nt0;
    cp_async_wait<1>();
    __syncwarp();
    const uint32_t kb_s = wbase_s + st * 2 * kKvTile, vb_s = kb_s + kKvTile;

    // S = Q K^T over the page's 16 tokens (two n-tiles of 8)
    float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
    {
      const int mi = lane >> 3, ri = lane & 7;
      const int tok = (mi >> 1) * 8 + ri;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        uint32_t kb[4];
        ldmatrix_x4(kb, kb_s + swz(tok, 2 * kk + (mi & 1)));
        mma_bf16(s0, qa[kk], kb[0], kb[1]);
        mma_bf16(s1, qa[kk], kb[2], kb[3]);
      }
    }
    // online softmax in base 2; token of s0[0..1] = 2t4, 2t4+1; s1: +8
    const int tk0 = 2 * t4, tk1 = 2 * t4 + 1, tk2 = 8 + 2 * t4, tk3 = 9 + 2 * t4;
    float x0 = tk0 < ntok ? s0[0] * kDecScale : -INFINITY;
    float x1 = tk1 < ntok ? s0[1] * kDecScale : -INFINITY;
    float x2 = tk2 < ntok ? s1[0] * kDecScale : -INFINITY;
    float x3 = tk3 < ntok ? s1[1] * kDecScale : -INFINITY;
    float mx = fmaxf(fmaxf(x0, x1), fmaxf(x2, x3));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float m_new = fmaxf(m_run, mx);
    const float corr = exp2f(m_run - m_new);
    const float p0 = exp2f(x0 - m_new), p1 = exp2f(x1 - m_new);
    const float p2 = exp2f(x2 - m_new), p3 = exp2f(x3 - m_new);
    l_run = l_run * corr + (p0 + p1 + p2 + p3);
    m_run = m_new;
    float corr8 = 1.f, p80 = 0.f, p81 = 0.f, p82 = 0.f, p83 = 0.f;
    if (WIDE) {
      const float y0 = tk0 < ntok ? s0[2] * kDecScale : -INFINITY;
      const float y1 = tk1 < ntok ? s0[3] * kDecScale : -INFINITY;
      const float y2 = tk2 < ntok ? s1[2] * kDecScale : -INFINITY;
      const float y3 = tk3 < ntok ? s1[3] * kDecScale : -INFINITY;
      float my = fmaxf(fmaxf(y0, y1), fmaxf(y2, y3));
      my = fmaxf(my, __shfl_xor_sync(0xffffffffu, my, 1));
      my = fmaxf(my, __shfl_xor_sync(0xffffffffu, my, 2));
      const float m8 = fmaxf(m_run8, my);
      corr8 = exp2f(m_run8 - m8);
      p80 = exp2f(y0 - m8);
      p81 = exp2f(y1 - m8);
      p82 = exp2f(y2 - m8);
      p83 = exp2f(y3 - m8);
      l_run8 = l_run8 * corr8 + (p80 + p81 + p82 + p83);
      m_run8 = m8;
    }
    uint32_t pa[4];
    pa[0] = pack_bf2(p0, p1);
    pa[1] = pack_bf2(p80, p81);
    pa[2] = pack_bf2(p2, p3);
    pa[3] = pack_bf2(p82, p83);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      o[i][0] *= corr;
      o[i][1] *= corr;
      o[i][2] *= corr8;
      o[i][3] *= corr8;
    }
    // O += P V (16 n-tiles of 8 head dims)
    {
      const int mi = lane >> 3, ri = lane & 7;
      const int tok = (mi & 1) * 8 + ri;
#pragma unroll
      for (int nd = 0; nd < 8; ++nd) {
        uint32_t vb[4];
        ldmatrix_x4_trans(vb, vb_s + swz(tok, 2 * nd + (mi >> 1)));
        mma_bf16(o[2 * nd], pa, vb[0], vb[1]);
        mma_bf16(o[2 * nd + 1], pa, vb[2], vb[3]);
      }
    }
    __syncwarp();
    if (st) {
      have1 = fetch_next(ph1, nt1);
      if (have1) issue(1, ph1);
    } else {
      have0 = fetch_next(ph0, nt0);
      if (have0) issue(0, ph0);
    }
    cp_async_commit();
  }
  cp_async_wait<0>();
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
  l_run8 += __shfl_xor_sync(0xffffffffu, l_run8, 1);
  l_run8 += __shfl_xor_sync(0xffffffffu, l_run8, 2);
  __syncthreads();

  // merge the four warps: smem [warp][16 rows][128] + m, l
  float *sO = reinterpret_cast<float *>(smem);
  float *sM = sO + kDecWarps * 16 * kDim;
  float *sL = sM + kDecWarps * 16;
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) {
    const int d = nt * 8 + 2 * t4;
    sO[(wid * 16 + gq) * kDim + d] = o[nt][0];
    sO[(wid * 16 + gq) * kDim + d + 1] = o[nt][1];
    sO[(wid * 16 + gq + 8) * kDim + d] = o[nt][2];
    sO[(wid * 16 + gq + 8) * kDim + d + 1] = o[nt][3];
  }
  if (t4 == 0) {
    sM[wid * 16 + gq] = m_run;
    sL[wid * 16 + gq] = l_run;
    sM[wid * 16 + gq + 8] = m_run8;
    sL[wid * 16 + gq + 8] = l_run8;
  }
  __syncthreads();
  const int d = threadIdx.x;  // 128 threads = head dim
  for (int g = 0; g < G; ++g) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, sM[w * 16 + g]);
    float Lsum = 0.f, acc = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) {
        const float mw = sM[w * 16 + g];
        if (mw == -INFINITY) continue;
        const float f = exp2f(mw - M);
        Lsum += sL[w * 16 + g] * f;
        acc += sO[(w * 16 + g) * kDim + d] * f;
      }
    }
    const float ov = Lsum > 0.f ? acc / Lsum : 0.f;
    const float lse = Lsum > 0.f ? (M + log2f(Lsum)) * kLn2f : -INFINITY;
    const size_t row = (size_t)b * h_q + (size_t)h * G + g;
    if (n_split == 1) {
      o_out[row * kDim + d] = __float2bfloat16_rn(ov);
      if (d == 0) lse_out[row] = lse;
    } else {
      o_part[(row * n_split + split) * kDim + d] = ov;
      if (d == 0) lse_part[row * n_split + split] = lse;
    }
  }
}

__global__ void __launch_bounds__(kDim)
    combine_kernel(const float *__restrict__ o_part,
                   const float *__restrict__ lse_part, int n_split,
                   __nv_bfloat16 *__restrict__ o_out,
                   float *__restrict__ lse_out) {
  const size_t row = blockIdx.x;
  const int d = threadIdx.x;
  const float *lp = lse_part + row * n_split;
  float M = -INFINITY;
  for (int s = 0; s < n_split; ++s) M = fmaxf(M, lp[s]);
  float wsum = 0.f, acc = 0.f;
  if (M != -INFINITY) {
    for (int s = 0; s < n_split; ++s) {
      if (lp[s] == -INFINITY) continue;
      const float w = expf(lp[s] - M);
      wsum += w;
      acc += w * o_part[(row * n_split + s) * kDim + d];
    }
  }
  o_out[row * kDim + d] = __float2bfloat16_rn(wsum > 0.f ? acc / wsum : 0.f);
  if (d == 0) lse_out[row] = wsum > 0.f ? M + logf(wsum) : -INFINITY;
}

// --------------------------------------------------------------------------
// launchers
// --------------------------------------------------------------------------
static int dec_sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

int decode_pages_per_split(int list_len, long long units) {
  const int sms = dec_sm_count();
  int pps = 16;
  while (pps < list_len && (list_len + pps - 1) / pps > kMaxSplits) pps *= 2;
  while (pps > 4 && units * ((list_len + pps - 1) / pps) < 4LL * sms &&
         (list_len + pps / 2 - 1) / (pps / 2) <= kMaxSplits)
    pps /= 2;
  return pps;
}

cudaError_t launch_decode(const void *q, const void *k_cache,
                          const void *v_cache, int64_t num_phys,
                          const int32_t *pt, const int32_t *seq_lens,
                          const int32_t *idx, int k, int batch, int h_kv,
                          int G, int max_pages, void *o_out, float *lse_out,
                          float *o_part, float *lse_part, int32_t *status,
                          cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(
        decode_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
        227 * 1024);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(decode_kernel<true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             227 * 1024);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int list_len = idx ? k : max_pages;
  const int pps = decode_pages_per_split(list_len, (long long)batch * h_kv);
  const int n_split = (list_len + pps - 1) / pps;
  const size_t smem = kDecSmem + 2 * sizeof(int) * (size_t)pps;
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  dim3 grid(n_split, h_kv, batch);
  auto *qq = static_cast<const __nv_bfloat16 *>(q);
  auto *kc = static_cast<const __nv_bfloat16 *>(k_cache);
  auto *vc = static_cast<const __nv_bfloat16 *>(v_cache);
  auto *oo = static_cast<__nv_bfloat16 *>(o_out);
  if (G > 8)
    decode_kernel<true><<<grid, kDecThreads, smem, stream>>>(
        qq, kc, vc, num_phys, pt, seq_lens, idx, k, h_kv, G, max_pages, pps,
        n_split, oo, lse_out, o_part, lse_part, status);
  else
    decode_kernel<false><<<grid, kDecThreads, smem, stream>>>(
        qq, kc, vc, num_phys, pt, seq_lens, idx, k, h_kv, G, max_pages, pps,
        n_split, oo, lse_out, o_part, lse_part, status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || n_split == 1) return e;
  combine_kernel<<<(unsigned)((size_t)batch * h_kv * G), kDim, 0, stream>>>(
      o_part, lse_part, n_split, oo, lse_out);
  return cudaGetLastError();
}

}  // namespace locks
