// GQA-shared page selection (LOCKS reading notes §4.2 Eq.(5) with the
// sink/recent rule, §4.4 Algorithm 2): per (sequence, KV head), normalise
// each head's page scores into mass fractions, average them over the group
// and keep the sink page, the recent page and the k-2 other pages of largest
// share (ties to the lower page).
#include "common.cuh"
#include "launch.h"

namespace locks {

// ---------------------------------------------------------------------------
// selection: one CTA per (sequence, KV head)
// ---------------------------------------------------------------------------
constexpr int kSelThreads = 512;

__device__ __forceinline__ uint32_t order_key(float x) {
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Sum of the per-warp values v[0..wid) (one per warp of the block, in
// shared memory): a shuffle scan over the warps instead of a loop
template <int NWARPS>
__device__ __forceinline__ int warps_before(const int *v, int wid, int lane) {
  const int x = lane < NWARPS ? v[lane] : 0;
  int incl = x;
#pragma unroll
  for (int o = 1; o < NWARPS; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  return __shfl_sync(0xffffffffu, incl - x, wid);
}

// block-wide exclusive scan of two counters (blockDim = kSelThreads)
__device__ __forceinline__ void block_scan2(int a, int b, int &ea, int &eb,
                                            int *sh /* [2*32] */) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int ia = a, ib = b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int va = __shfl_up_sync(0xffffffffu, ia, o);
    const int vb = __shfl_up_sync(0xffffffffu, ib, o);
    if (lane >= o) {
      ia += va;
      ib += vb;
    }
  }
  if (lane == 31) {
    sh[wid] = ia;
    sh[32 + wid] = ib;
  }
  __syncthreads();
  if (wid == 0) {
    const int nw = (int)(blockDim.x >> 5);
    int wa = lane < nw ? sh[lane] : 0, wb = lane < nw ? sh[32 + lane] : 0;
    int sa = wa, sb = wb;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int va = __shfl_up_sync(0xffffffffu, sa, o);
      const int vb = __shfl_up_sync(0xffffffffu, sb, o);
      if (lane >= o) {
        sa += va;
        sb += vb;
      }
    }
    sh[lane] = sa - wa;
    sh[32 + lane] = sb - wb;
  }
  __syncthreads();
  ea = sh[wid] + ia - a;
  eb = sh[32 + wid] + ib - b;
  __syncthreads();
}

// Scores of pages j0..j0+3 of every head of the group; pages at or past
// `lim` read as `fill`.
template <int GT>
__device__ __forceinline__ void load_quad(const float *sc, int max_pages,
                                          int G, bool vec, int j0, int lim,
                                          float fill, float (&x)[GT][4]) {
#pragma unroll
  for (int g = 0; g < GT; ++g) {
    const float *row = sc + (size_t)g * max_pages;
    if (g < G && vec && j0 + 3 < lim) {
      const float4 v = __ldg(reinterpret_cast<const float4 *>(row + j0));
      x[g][0] = v.x;
      x[g][1] = v.y;
      x[g][2] = v.z;
      x[g][3] = v.w;
    } else {
#pragma unroll
      for (int u = 0; u < 4; ++u)
        x[g][u] = (g < G && j0 + u < lim) ? __ldg(row + j0 + u) : fill;
    }
  }
}

// Keys j0..j0+3 (16-byte aligned when `kvec`); keys at or past `lim` read 0.
__device__ __forceinline__ uint4 load_keys4(const uint32_t *keys, int j0,
                                            int lim, bool kvec) {
  if (kvec && j0 + 3 < lim) return *reinterpret_cast<const uint4 *>(keys + j0);
  uint4 v;
  v.x = j0 < lim ? keys[j0] : 0u;
  v.y = j0 + 1 < lim ? keys[j0 + 1] : 0u;
  v.z = j0 + 2 < lim ? keys[j0 + 2] : 0u;
  v.w = j0 + 3 < lim ? keys[j0 + 3] : 0u;
  return v;
}

// Keys live in shared memory when they fit (SMEM_KEYS), else in the
// workspace.  Keys are indexed by page; the sink, the recent page and pages
// past the candidates hold key 0, which is below every real key.
constexpr int kRadixBits = 12;
constexpr int kRadixBins = 1 << kRadixBits;
constexpr int kBinsPerWarp = kRadixBins / (kSelThreads / 32);  // 256

// MINB: resident CTAs per SM the registers are sized for.  2 when there are
// more (sequence, KV head) units than SMs; 1 when every unit has an SM of
// its own, which leaves registers for more pages in flight per thread.
template <bool SMEM_KEYS, int GT, int MINB>
__global__ void __launch_bounds__(kSelThreads, MINB)
    select_kernel(const float *__restrict__ scores,
                  const int32_t *__restrict__ seq_lens, int h_kv, int G,
                  int max_pages, int k, int rule,
                  int32_t *__restrict__ idx, uint32_t *__restrict__ keybuf,
                  int32_t *status) {
  extern __shared__ __align__(16) uint32_t sel_keys[];
  __shared__ float zs[kMaxGroup];
  __shared__ float red_m[32][kMaxGroup], red_s[32][kMaxGroup];
  __shared__ __align__(16) int hist[2][kRadixBins];
  __shared__ int sh_wcnt[2][32];
  __shared__ uint32_t red_u[2][32];
  __shared__ uint32_t sh_prefix, sh_mask;
  __shared__ int sh_remaining, sh_varying, sh_slow;

  const int b = blockIdx.y, h = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  constexpr int nwarps = kSelThreads / 32;
  pdl_trigger();
  int L = seq_lens[b];
  if (L < 0 || L > max_pages * kPage) {
    if (tid == 0 && h == 0) set_status(status, LOCKS_DEV_BAD_SEQ_LEN);
    L = max(0, min(L, max_pages * kPage));
  }
  const int n = (L + kPage - 1) / kPage, nf = L / kPage;
  int32_t *out = idx + ((size_t)b * h_kv + h) * k;
  pdl_wait();  // scores of the scoring kernel; idx may still be read before
  if (n <= k) {
    for (int i = tid; i < k; i += blockDim.x) out[i] = i < n ? i : -1;
    return;
  }
  if (k == 2) {  // only the sink and the recent page
    if (tid == 0) {
      out[0] = 0;
      out[1] = n - 1;
    }
    return;
  }
  const float *sc = scores + ((size_t)b * h_kv + h) * G * (size_t)max_pages;
  uint32_t *keys = SMEM_KEYS
                       ? sel_keys
                       : keybuf + ((size_t)b * h_kv + h) * (size_t)max_pages;
  constexpr float kLog2e = 1.4426950408889634f;
  // pages are read four at a time when every row starts 16-byte aligned
  const bool vec = (max_pages & 3) == 0 &&
                   ((reinterpret_cast<uintptr_t>(scores) & 15u) == 0);
  const bool kvec = SMEM_KEYS || (max_pages & 3) == 0;  // 16-byte key rows
  const int nq = (n + 3) >> 2;        // quads of pages covering [0, n)
  // quads a thread has in flight at once (what the registers allow)
  // (at two CTAs per SM and G = 4 a second quad in flight measured slower,
  // 16.6 against 16.2 us on 256 units, and spilled)
  constexpr int R = MINB == 1 ? (GT <= 8 ? 2 : 1) : (GT <= 2 ? 2 : 1);
  for (int i = tid; i < kRadixBins; i += blockDim.x) hist[0][i] = 0;

  // Z_g: log2-sum-exp2 over the summarised pages [0, nf) (group-mass
  // pooling does not normalise per head and skips it).  Common form: every
  // thread sums 2^(x - r_g) against one reference per head, r_g = the score
  // of page 0 (always summarised here, since n > k >= 2), so the block
  // combine is a plain sum; a score more than 2^7 above r_g (the sum
  // overflows) or a page-0 score that is not finite takes the general form
  // below, with per-thread references.
  if (rule != LOCKS_MERGE_GROUP_MASS) {
  float ref[GT];
  bool finite = true;
#pragma unroll
  for (int g = 0; g < GT; ++g) {
    ref[g] = g < G ? __ldg(sc + (size_t)g * max_pages) * kLog2e : 0.f;
    finite = finite && !(fabsf(ref[g]) > 3.0e38f) && ref[g] == ref[g];
  }
  if (tid == 0) sh_slow = 0;
  if (finite) {
    float s[GT];
#pragma unroll
    for (int g = 0; g < GT; ++g) s[g] = 0.f;
    for (int qd = tid; qd < nq; qd += R * blockDim.x) {
      float x[R][GT][4];
#pragma unroll
      for (int r = 0; r < R; ++r)
        load_quad<GT>(sc, max_pages, G, vec, 4 * (qd + r * blockDim.x), nf,
                      -INFINITY, x[r]);
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int g = 0; g < GT; ++g)
#pragma unroll
          for (int u = 0; u < 4; ++u)
            s[g] += ex2_fast(fmaf(x[r][g][u], kLog2e, -ref[g]));
    }
#pragma unroll
    for (int g = 0; g < GT; ++g) {
      float sg = s[g];
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1)
        sg += __shfl_xor_sync(0xffffffffu, sg, o);
      if (lane == 0) red_s[wid][g] = sg;
    }
    __syncthreads();
    if (tid < G) {
      float sum = 0.f;
      for (int w = 0; w < nwarps; ++w) sum += red_s[w][tid];
      zs[tid] = __ldg(sc + (size_t)tid * max_pages) * kLog2e + lg2_fast(sum);
      if (!(sum < INFINITY)) sh_slow = 1;
    }
    __syncthreads();
  }
  if (!finite || sh_slow) {
  {
    float m[GT], s[GT];
#pragma unroll
    for (int g = 0; g < GT; ++g) {
      m[g] = -INFINITY;
      s[g] = 0.f;
    }
    // Each thread sums 2^(x - m_g) against its own reference m_g, raised
    // (and the sum rescaled) only when a quad's maximum passes it by more
    // than 2^6, so the common step is one exponential per score; terms stay
    // below 2^64 and the sum below 2^77.
    for (int qd = tid; qd < nq; qd += R * blockDim.x) {
      float x[R][GT][4];
#pragma unroll
      for (int r = 0; r < R; ++r)
        load_quad<GT>(sc, max_pages, G, vec, 4 * (qd + r * blockDim.x), nf,
                      -INFINITY, x[r]);
#pragma unroll
      for (int r = 0; r < R; ++r) {
#pragma unroll
        for (int g = 0; g < GT; ++g) {
          if (g >= G) continue;
          const float cm = fmaxf(fmaxf(x[r][g][0], x[r][g][1]),
                                 fmaxf(x[r][g][2], x[r][g][3])) * kLog2e;
          if (cm > m[g] + 64.f) {  // also the first finite score
            s[g] = m[g] == -INFINITY ? 0.f : s[g] * ex2_fast(m[g] - cm);
            m[g] = cm;
          }
          const float ref = m[g] == -INFINITY ? 0.f : m[g];
#pragma unroll
          for (int u = 0; u < 4; ++u)
            s[g] += ex2_fast(fmaf(x[r][g][u], kLog2e, -ref));
        }
      }
    }
#pragma unroll
    for (int g = 0; g < GT; ++g) {
      float mg = m[g], sg = s[g];
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, mg, o);
        const float s2 = __shfl_xor_sync(0xffffffffu, sg, o);
        const float mm = fmaxf(mg, m2);
        sg = (mg == -INFINITY ? 0.f : sg * ex2_fast(mg - mm)) +
             (m2 == -INFINITY ? 0.f : s2 * ex2_fast(m2 - mm));
        mg = mm;
      }
      if (lane == 0 && g < G) {
        red_m[wid][g] = mg;
        red_s[wid][g] = sg;
      }
    }
  }
  __syncthreads();
  if (tid < G) {
    float m = -INFINITY;
    for (int w = 0; w < nwarps; ++w) m = fmaxf(m, red_m[w][tid]);
    float s = 0.f;
    for (int w = 0; w < nwarps; ++w)
      if (red_m[w][tid] != -INFINITY)
        s += red_s[w][tid] * ex2_fast(red_m[w][tid] - m);
    zs[tid] = m + lg2_fast(s);
  }
  __syncthreads();
  }
  } else {
    if (tid < G) zs[tid] = 0.f;
    __syncthreads();
  }

  // key of page j (candidates 1..n-2), in base 2: share-average
  // log2 sum_g 2^(s_gj - Z_g) (each term <= 1 since Z_g bounds every
  // score), group-mass log2 sum_g 2^(s_gj) (Z_g = 0 above), group-max
  // max_g (s_gj - Z_g)
  uint32_t kmin = 0xffffffffu, kmax = 0u;
  float zreg[GT];
#pragma unroll
  for (int g = 0; g < GT; ++g) zreg[g] = g < G ? zs[g] : 0.f;
  // last block of quads first: the normaliser pass just read them, so the
  // part of the scores still in L1 is read before it is evicted
  const int qstep = R * blockDim.x;
  for (int it = (nq + qstep - 1) / qstep - 1; it >= 0; --it) {
    const int qd = it * qstep + tid;
    if (qd >= nq) continue;
    float x[R][GT][4];
    // heads at or above G read -inf: no term, no maximum
#pragma unroll
    for (int r = 0; r < R; ++r)
      load_quad<GT>(sc, max_pages, G, vec, 4 * (qd + r * blockDim.x), nf,
                    -INFINITY, x[r]);
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int j0 = 4 * (qd + r * blockDim.x);
      if (j0 >= 4 * nq) break;
      uint32_t kq[4];
      float key[4];
      if (rule == LOCKS_MERGE_GROUP_MAX) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          key[u] = -INFINITY;
#pragma unroll
          for (int g = 0; g < GT; ++g)
            key[u] = fmaxf(key[u], fmaf(x[r][g][u], kLog2e, -zreg[g]));
        }
      } else {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          float sum = 0.f;
#pragma unroll
          for (int g = 0; g < GT; ++g)
            sum += ex2_fast(fmaf(x[r][g][u], kLog2e, -zreg[g]));
          key[u] = lg2_fast(sum);
          if (!(sum > 0.f && sum < INFINITY)) {
            // every term underflowed (or, pooling raw masses, overflowed):
            // subtract the largest first
            float m = -INFINITY;
#pragma unroll
            for (int g = 0; g < GT; ++g)
              m = fmaxf(m, fmaf(x[r][g][u], kLog2e, -zreg[g]));
            float t = 0.f;
#pragma unroll
            for (int g = 0; g < GT; ++g)
              t += ex2_fast(fmaf(x[r][g][u], kLog2e, -zreg[g]) - m);
            key[u] = m + lg2_fast(t);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        // candidates are pages 1..n-2
        const bool cand = (unsigned)(j0 + u - 1) <= (unsigned)(n - 3);
        kq[u] = cand ? order_key(key[u]) : 0u;
        kmin = min(kmin, cand ? kq[u] : 0xffffffffu);
        kmax = max(kmax, kq[u]);
      }
      if (kvec) {
        *reinterpret_cast<uint4 *>(keys + j0) =
            make_uint4(kq[0], kq[1], kq[2], kq[3]);
      } else {
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (j0 + u < n) keys[j0 + u] = kq[u];
      }
    }
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
    kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
  }
  if (lane == 0) {
    red_u[0][wid] = kmin;
    red_u[1][wid] = kmax;
  }
  __syncthreads();
  if (tid == 0) {
    uint32_t a = 0xffffffffu, z = 0u;
    for (int w = 0; w < nwarps; ++w) {
      a = min(a, red_u[0][w]);
      z = max(z, red_u[1][w]);
    }
    // bits above the highest one where min and max differ are common to
    // every candidate key
    const int varying = (a == z) ? 0 : 32 - __clz(a ^ z);
    const uint32_t msk = varying == 32 ? 0u : ~((1u << varying) - 1u);
    sh_prefix = z & msk;
    sh_mask = msk;
    sh_remaining = k - 2;
    sh_varying = varying;
  }
  __syncthreads();

  // radix select of the (k-2)-th largest key over the varying bits,
  // 12-bit digits from the top; key 0 never matches a candidate prefix.
  // Histograms alternate between two buffers so the next one is cleared
  // while the current one fills.
  const int varying = sh_varying;
  const int nk4 = (n + 3) >> 2;
  for (int top = varying, pass = 0; top > 0; top -= kRadixBits, ++pass) {
    const int width = min(kRadixBits, top), shift = top - width;
    const uint32_t dmask = (1u << width) - 1u;
    int *hc = hist[pass & 1];
    int *hn = hist[(pass & 1) ^ 1];
    const uint32_t pre = sh_prefix, msk = sh_mask;
    const int rem = sh_remaining;
    for (int i = tid; i < kRadixBins; i += blockDim.x) hn[i] = 0;
    for (int qd = tid; qd < nk4; qd += blockDim.x) {
      const uint4 v = load_keys4(keys, 4 * qd, n, kvec);
      const uint32_t kv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (kv[u] != 0u && (kv[u] & msk) == pre)
          atomicAdd(&hc[(kv[u] >> shift) & dmask], 1);
    }
    __syncthreads();
    // warp w covers digits [bins-256(w+1), bins-256w), lane l its eight
    // digits from the top; counts are scanned from the largest digit down
    const int hi = kRadixBins - 1 - kBinsPerWarp * wid - 8 * lane;
    const int4 c4 = *reinterpret_cast<const int4 *>(hc + hi - 3);
    const int4 d4 = *reinterpret_cast<const int4 *>(hc + hi - 7);
    const int cnt = c4.x + c4.y + c4.z + c4.w + d4.x + d4.y + d4.z + d4.w;
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) sh_wcnt[0][wid] = incl;
    __syncthreads();
    const int before = warps_before<nwarps>(sh_wcnt[0], wid, lane);
    const int mine = before + incl - cnt;  // count above this lane's digits
    if (mine < rem && rem <= mine + cnt) {
      const int c[8] = {c4.w, c4.z, c4.y, c4.x,
                        d4.w, d4.z, d4.y, d4.x};  // digits hi, hi-1, ...
      int acc = mine;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (acc < rem && rem <= acc + c[i]) {
          sh_prefix = pre | ((uint32_t)(hi - i) << shift);
          sh_mask = msk | (dmask << shift);
          sh_remaining = rem - acc;
        }
        acc += c[i];
      }
    }
    __syncthreads();
  }
  const uint32_t T = sh_prefix;
  const int need_eq = sh_remaining;  // keys equal to T to keep (lowest j)

  // ordered compaction: warp w owns pages [w*seg, (w+1)*seg), walked 128 at
  // a time (four per lane); warps' counts are scanned once
  const int seg = ((n + nwarps - 1) / nwarps + 127) & ~127;
  const int w_lo = min(n, wid * seg), w_hi = min(n, w_lo + seg);
  int gt = 0, eq = 0;
  for (int j0 = w_lo + 4 * lane; j0 < w_hi; j0 += 128) {
    const uint4 v = load_keys4(keys, j0, w_hi, kvec);
    gt += (v.x > T) + (v.y > T) + (v.z > T) + (v.w > T);
    eq += (v.x == T) + (v.y == T) + (v.z == T) + (v.w == T);
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    gt += __shfl_xor_sync(0xffffffffu, gt, o);
    eq += __shfl_xor_sync(0xffffffffu, eq, o);
  }
  int gt_before, eq_before;
  if constexpr (SMEM_KEYS) {
    // n <= 32768 pages: both counts and their sums stay below 2^15
    if (lane == 0) sh_wcnt[0][wid] = (eq << 16) | gt;
    __syncthreads();
    const int ge_before = warps_before<nwarps>(sh_wcnt[0], wid, lane);
    gt_before = ge_before & 0xffff;
    eq_before = ge_before >> 16;
  } else {
    if (lane == 0) {
      sh_wcnt[0][wid] = gt;
      sh_wcnt[1][wid] = eq;
    }
    __syncthreads();
    gt_before = warps_before<nwarps>(sh_wcnt[0], wid, lane);
    eq_before = warps_before<nwarps>(sh_wcnt[1], wid, lane);
  }
  for (int base = w_lo; base < w_hi; base += 128) {
    const int j0 = base + 4 * lane;
    const uint4 v = load_keys4(keys, j0, w_hi, kvec);
    const uint32_t kv[4] = {v.x, v.y, v.z, v.w};
    int ngt = 0, neq = 0;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      ngt += kv[u] > T;
      neq += kv[u] == T;
    }
    // most groups of 128 hold no key at or above the threshold
    if (!__any_sync(0xffffffffu, ngt + neq > 0)) continue;
    // exclusive scan of (eq << 16 | gt) over the lanes
    const int packed = (neq << 16) | ngt;
    int incl = packed;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    const int tot = __shfl_sync(0xffffffffu, incl, 31);
    int my_gt = gt_before + ((incl - packed) & 0xffff);
    int my_eq = eq_before + ((incl - packed) >> 16);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const bool is_gt = kv[u] > T, is_eq = kv[u] == T;
      if (is_gt || (is_eq && my_eq < need_eq)) {
        const int pos = 1 + my_gt + min(my_eq, need_eq);
        if (pos >= 1 && pos < k - 1)
          out[pos] = j0 + u;
        else
          set_status(status, LOCKS_DEV_BAD_INDEX);
      }
      my_gt += is_gt;
      my_eq += is_eq;
    }
    gt_before += tot & 0xffff;
    eq_before += tot >> 16;
  }
  if (tid == 0) {
    out[0] = 0;
    out[k - 1] = n - 1;
  }
}

// --------------------------------------------------------------------------
// launcher
// --------------------------------------------------------------------------
constexpr int kSelSmemKeys = 32 * 1024;   // candidate keys held on chip

cudaError_t launch_select(const float *scores, const int32_t *seq_lens,
                          int batch, int h_kv, int G, int max_pages, int k,
                          int rule, int32_t *idx, uint32_t *keybuf,
                          int32_t *status, cudaStream_t stream) {
  dim3 grid(h_kv, batch);
  const bool on_chip = max_pages <= kSelSmemKeys;
  const size_t smem = on_chip ? (size_t)((max_pages + 3) & ~3) * 4 : 0;
  auto run = [&](auto kern) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(
        kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSelSmemKeys * 4);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, grid, dim3(kSelThreads), smem, stream, scores,
                      seq_lens, h_kv, G, max_pages, k, rule, idx, keybuf,
                      status);
  };
  const int gt = G <= 1 ? 1 : G <= 2 ? 2 : G <= 4 ? 4 : G <= 8 ? 8 : 16;
  // one CTA per SM suffices when the units fit the GPU in one wave
  const bool own_sm = (long long)batch * h_kv <= device_sm_count();
  // G > 8 always runs the one-CTA-per-SM form: with two per SM its
  // registers spill (on 256 units of 8,192 pages, 74 us against 50 us)
#define LOCKS_SELECT_CASES(SK, MB)                         \
  switch (gt) {                                            \
    case 1: return run(select_kernel<SK, 1, MB>);          \
    case 2: return run(select_kernel<SK, 2, MB>);          \
    case 4: return run(select_kernel<SK, 4, MB>);          \
    case 8: return run(select_kernel<SK, 8, MB>);          \
    default: return run(select_kernel<SK, 16, 1>);         \
  }
  if (on_chip) {
    if (own_sm) LOCKS_SELECT_CASES(true, 1)
    LOCKS_SELECT_CASES(true, 2)
  }
  if (own_sm) LOCKS_SELECT_CASES(false, 1)
  LOCKS_SELECT_CASES(false, 2)
#undef LOCKS_SELECT_CASES
}

}  // namespace locks
