// Exact page log-sum-exp (LOCKS reading notes §4.2 Eq.(4) and §6 Fig. 1(b),
// Fig. 2): s_j(q_g) = ln sum_{i < 16} exp(q_g . k_i / sqrt(d)) for every full
// page j of every (sequence, KV head) and every query head g of the group --
// the quantity the page summaries estimate.  Ranking pages by it is the
// exact-mass selector the notes compare LOCKS against; it reads every key.
//
// Same streaming scheme as the sparse decode: the full pages of all
// (sequence, KV head) units are laid end to end and cut into equal
// contiguous runs, one per warp.  A warp resolves 32 pages at a time through
// the page table, gathers each page's 4 KB of keys with 16-byte cp.async
// into a double-buffered, XOR-swizzled shared-memory tile, and computes the
// group's 16 logits per head with bf16 mma.sync (heads as the M dimension),
// then the log-sum-exp in base 2.
#include "common.cuh"
#include "launch.h"

namespace locks {

constexpr int kExWarps = 4;
constexpr int kExThreads = 32 * kExWarps;
constexpr int kExStages = 2;
constexpr int kExTile = kPage * kDim * 2;                 // 4096 bytes
constexpr int kExRing = kExWarps * kExStages * kExTile;  // 32 KB
constexpr float kExScale = 0.12751743074602467f;         // log2(e)/sqrt(d)
constexpr float kExLn2 = 0.69314718055994531f;

// swizzled byte offset of 16-byte chunk `ch` (0..15) of token row `row`
__device__ __forceinline__ uint32_t ex_swz(int row, int ch) {
  return (uint32_t)(row * 256 + ((ch ^ (row & 7)) << 4));
}

template <bool WIDE>
__global__ void __launch_bounds__(kExThreads)
    exact_kernel(const __nv_bfloat16 *__restrict__ q,
                 const __nv_bfloat16 *__restrict__ k_cache, int64_t num_phys,
                 const int32_t *__restrict__ pt,
                 const int32_t *__restrict__ seq_lens, int batch, int h_kv,
                 int G, int max_pages, int n_warps,
                 float *__restrict__ scores, int32_t *status) {
  extern __shared__ __align__(128) uint8_t smem[];
  int *s_pre = reinterpret_cast<int *>(smem + kExRing);  // [batch + 1]
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int gq = lane >> 2, t4 = lane & 3;
  const int h_q = h_kv * G;

  // positions per sequence: h_kv lists of its full pages; inclusive scan
  for (int b = threadIdx.x; b < batch; b += blockDim.x) {
    int L = seq_lens[b];
    if (L < 0 || L > max_pages * kPage) {
      if (blockIdx.x == 0) set_status(status, LOCKS_DEV_BAD_SEQ_LEN);
      L = max(0, min(L, max_pages * kPage));
    }
    s_pre[b + 1] = h_kv * (L / kPage);
  }
  if (threadIdx.x == 0) s_pre[0] = 0;
  __syncthreads();
  if (wid == 0) {
    const int per = (batch + 31) / 32;
    const int lo = 1 + lane * per, hi = min(batch + 1, lo + per);
    int run = 0;
    for (int i = lo; i < hi; ++i) {
      run += s_pre[i];
      s_pre[i] = run;
    }
    int incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    const int excl = incl - run;
    for (int i = lo; i < hi; ++i) s_pre[i] += excl;
  }
  __syncthreads();
  const int total = s_pre[batch];
  const int chunk = max(1, (total + n_warps - 1) / n_warps);
  const int gw = blockIdx.x * kExWarps + wid;
  if (gw >= n_warps || (long long)gw * chunk >= total) return;
  const int pb = gw * chunk, pe = min(total, pb + chunk);

  // position -> (unit, page): largest b with s_pre[b] <= p, then h, j
  auto locate = [&](int p, int &u, int &j) {
    int lo = 0, hi = batch;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_pre[mid] <= p) lo = mid; else hi = mid;
    }
    const int nf = (s_pre[lo + 1] - s_pre[lo]) / h_kv;
    const int r = p - s_pre[lo];
    const int h = r / nf;
    u = lo * h_kv + h;
    j = r - h * nf;
  };

  const uint32_t wbase_s = smem_u32(smem + wid * (kExStages * kExTile));
  uint32_t qa[8][4];
  auto load_q = [&](int u) {
    const int b = u / h_kv, h = u - b * h_kv;
    const __nv_bfloat16 *qb = q + ((size_t)b * h_q + (size_t)h * G) * kDim;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      const int d0 = 16 * s + 2 * t4;
      qa[s][0] = gq < G ? __ldg(reinterpret_cast<const uint32_t *>(qb + gq * kDim + d0)) : 0u;
      qa[s][2] = gq < G ? __ldg(reinterpret_cast<const uint32_t *>(qb + gq * kDim + d0 + 8)) : 0u;
      qa[s][1] = (WIDE && gq + 8 < G) ? __ldg(reinterpret_cast<const uint32_t *>(qb + (gq + 8) * kDim + d0)) : 0u;
      qa[s][3] = (WIDE && gq + 8 < G) ? __ldg(reinterpret_cast<const uint32_t *>(qb + (gq + 8) * kDim + d0 + 8)) : 0u;
    }
  };

  // lane-resolved window of 32 positions: physical page (-1 if invalid),
  // unit and page of position win + lane
  int win = pb - 32, w_phys = -1, w_u = 0, w_j = 0;
  auto resolve = [&](int base) {
    const int p = base + lane;
    w_phys = -1;
    if (p < pe) {
      locate(p, w_u, w_j);
      const int b = w_u / h_kv;
      const int ph = __ldg(pt + (size_t)b * max_pages + w_j);
      if (ph < 0 || ph >= num_phys)
        set_status(status, LOCKS_DEV_BAD_PAGE_ID);
      else
        w_phys = ph;
    }
  };
  // item of position p (p in the current window): phys, unit, page
  auto item = [&](int p, int &phys, int &u, int &j) {
    if (p >= win + 32) {
      win += 32;
      resolve(win);
    }
    const int l = p - win;
    phys = __shfl_sync(0xffffffffu, w_phys, l);
    u = __shfl_sync(0xffffffffu, w_u, l);
    j = __shfl_sync(0xffffffffu, w_j, l);
  };
  auto issue = [&](int stage, int phys, int u) {
    if (phys >= 0) {
      const int h = u % h_kv;
      const uint8_t *ks = reinterpret_cast<const uint8_t *>(k_cache) +
                          ((size_t)phys * h_kv + h) * kExTile;
      const uint32_t kd = wbase_s + stage * kExTile;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int c = lane + 32 * i, row = c >> 4, ch = c & 15;
        cp_async16(kd + ex_swz(row, ch), ks + 16 * c);
      }
    }
    cp_async_commit();
  };

  int cur_u = -1;
  int ph0, u0, j0, ph1 = -1, u1 = 0, j1 = 0;
  item(pb, ph0, u0, j0);
  issue(0, ph0, u0);
  if (pb + 1 < pe) item(pb + 1, ph1, u1, j1);
  issue(1, pb + 1 < pe ? ph1 : -1, u1);

  for (int p = pb, st = 0; p < pe; ++p, st ^= 1) {
    const int phys = st ? ph1 : ph0, u = st ? u1 : u0, j = st ? j1 : j0;
    if (u != cur_u) {
      load_q(u);
      cur_u = u;
    }
    cp_async_wait<1>();
    __syncwarp();
    float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
    if (phys >= 0) {
      const uint32_t kb_s = wbase_s + st * kExTile;
      const int mi = lane >> 3, ri = lane & 7;
      const int tok = (mi >> 1) * 8 + ri;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        uint32_t kb[4];
        ldmatrix_x4(kb, kb_s + ex_swz(tok, 2 * kk + (mi & 1)));
        mma_bf16(s0, qa[kk], kb[0], kb[1]);
        mma_bf16(s1, qa[kk], kb[2], kb[3]);
      }
    }
    // rows gq (elements 0, 1) and gq + 8 (2, 3); tokens 2t4, 2t4+1 in s0,
    // 8 + 2t4, 9 + 2t4 in s1
#pragma unroll
    for (int half = 0; half < (WIDE ? 2 : 1); ++half) {
      const float x0 = s0[2 * half] * kExScale, x1 = s0[2 * half + 1] * kExScale;
      const float x2 = s1[2 * half] * kExScale, x3 = s1[2 * half + 1] * kExScale;
      float m = fmaxf(fmaxf(x0, x1), fmaxf(x2, x3));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
      float e = (exp2f(x0 - m) + exp2f(x1 - m)) + (exp2f(x2 - m) + exp2f(x3 - m));
      e += __shfl_xor_sync(0xffffffffu, e, 1);
      e += __shfl_xor_sync(0xffffffffu, e, 2);
      const int g = gq + 8 * half;
      if (t4 == 0 && g < G) {
        const float sv = phys >= 0 ? (m + log2f(e)) * kExLn2 : -INFINITY;
        scores[((size_t)cur_u * G + g) * max_pages + j] = sv;
      }
    }
    __syncwarp();
    // refill this stage with position p + 2
    int nph = -1, nu = 0, nj = 0;
    if (p + 2 < pe) item(p + 2, nph, nu, nj);
    issue(st, nph, nu);
    if (st) {
      ph1 = nph;
      u1 = nu;
      j1 = nj;
    } else {
      ph0 = nph;
      u0 = nu;
      j0 = nj;
    }
  }
  cp_async_wait<0>();
}

// --------------------------------------------------------------------------
// launcher
// --------------------------------------------------------------------------
size_t exact_smem_bytes(int batch) {
  return (size_t)kExRing + sizeof(int) * ((size_t)batch + 1);
}

int exact_max_batch() {
  return (int)((227 * 1024 - (size_t)kExRing - 64) / sizeof(int));
}

cudaError_t launch_exact(const void *q, const void *k_cache, int64_t num_phys,
                         const int32_t *pt, const int32_t *seq_lens,
                         int batch, int h_kv, int G, int max_pages,
                         float *scores, int32_t *status,
                         cudaStream_t stream) {
  static DeviceFlags attr_set, blocks_narrow, blocks_wide;
  cudaError_t ea = once_per_device(attr_set, [] {
    cudaError_t e = cudaFuncSetAttribute(
        exact_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
        227 * 1024);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(exact_kernel<true>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                227 * 1024);
  });
  if (ea != cudaSuccess) return ea;
  const size_t smem = exact_smem_bytes(batch);
  const int wide = G > 8 ? 1 : 0;
  const int blocks_per_sm =
      per_device_value(wide ? blocks_wide : blocks_narrow, [wide] {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                &n, wide ? exact_kernel<true> : exact_kernel<false>,
                kExThreads, exact_smem_bytes(64)) != cudaSuccess)
          return 0;
        return n;
      });
  long long warps = (long long)blocks_per_sm * device_sm_count() * kExWarps;
  const long long positions = (long long)batch * h_kv * max_pages;
  if (warps > positions) warps = positions;
  if (warps < 1) warps = 1;
  const int n_warps = (int)warps;
  const int grid = (n_warps + kExWarps - 1) / kExWarps;
  auto *qq = static_cast<const __nv_bfloat16 *>(q);
  auto *kc = static_cast<const __nv_bfloat16 *>(k_cache);
  if (wide)
    exact_kernel<true><<<grid, kExThreads, smem, stream>>>(
        qq, kc, num_phys, pt, seq_lens, batch, h_kv, G, max_pages, n_warps,
        scores, status);
  else
    exact_kernel<false><<<grid, kExThreads, smem, stream>>>(
        qq, kc, num_phys, pt, seq_lens, batch, h_kv, G, max_pages, n_warps,
        scores, status);
  return launched();
}

}  // namespace locks
