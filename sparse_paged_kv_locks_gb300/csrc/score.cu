// Summary scoring (LOCKS reading notes §4.2 Eq.(4)) and GQA-shared page
// selection (§4.2 Eq.(5) with the sink/recent rule, §4.4 Algorithm 2).
//
// Scoring streams the summary store, which is the dominant read of a decode
// step.  A persistent grid gives every warp a contiguous range of 8-record
// tiles (one (sequence, KV head) stream is contiguous); each warp double
// buffers its tiles in shared memory with 1-D bulk copies (TMA engine)
// completed on an mbarrier, and scores a tile with tensor-core mma.sync:
//   mma1  proj[g][n]  = sum_d q[g][d] V[d][n]            (8 k-steps / page)
//   mma2  L[g][i]     = sum_n proj[g][n] C[i][n]         (proj split in two
//                                                         fp16 halves)
//   mma3  qmu[g][p]   = sum_d q[g][d] mu_p[d]            (8 pages at once)
// Rows are the query heads of the group (M = 16 >= G), so every summary
// byte is read once for the whole GQA group.  Record bytes are laid out so
// each lane's mma fragments come from one 16-byte shared-memory read.
#include "common.cuh"
#include "launch.h"

namespace locks {

constexpr int kScoreWarps = 16;
constexpr int kScoreThreads = 32 * kScoreWarps;
constexpr int kTilePages = 8;
constexpr int kTileBytes = kTilePages * kRec;  // 6656
constexpr int kStages = 2;
constexpr int kRingBytes = kScoreWarps * kStages * kTileBytes;
// log2(e) / sqrt(128): logits are carried in base-2 units
constexpr float kLog2eRsqrtD = 0.12751743074602467f;
constexpr float kLn2 = 0.69314718055994531f;

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  return h2_as_u32(__floats2half2_rn(lo, hi));
}

__device__ __forceinline__ float lse2_quad(float a, float b, float c,
                                           float d) {
  float m = fmaxf(fmaxf(a, b), fmaxf(c, d));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
  float e = exp2f(a - m) + exp2f(b - m) + exp2f(c - m) + exp2f(d - m);
  e += __shfl_xor_sync(0xffffffffu, e, 1);
  e += __shfl_xor_sync(0xffffffffu, e, 2);
  return m + log2f(e);
}

struct TileInfo {
  int b, h, page0, npg;
};

// tile t -> (sequence, KV head, first page, pages) from the per-sequence
// prefix of tile counts (already multiplied by h_kv)
__device__ __forceinline__ TileInfo decode_tile(long long t, const int *prefix,
                                                const int *nfull, int batch,
                                                int h_kv) {
  int lo = 0, hi = batch;  // largest b with prefix[b] <= t
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= t) lo = mid; else hi = mid;
  }
  TileInfo ti;
  ti.b = lo;
  const int rem = (int)(t - prefix[lo]);
  const int tiles_b = (prefix[lo + 1] - prefix[lo]) / h_kv;
  ti.h = rem / tiles_b;
  const int j = rem - ti.h * tiles_b;
  ti.page0 = j * kTilePages;
  ti.npg = min(kTilePages, nfull[lo] - ti.page0);
  return ti;
}

template <bool WIDE>
__global__ void __launch_bounds__(kScoreThreads, 1)
    score_kernel(const __nv_bfloat16 *__restrict__ q,
                 const uint8_t *__restrict__ summaries,
                 const int32_t *__restrict__ seq_lens, int batch, int h_kv,
                 int G, int max_pages, float *__restrict__ s_hat,
                 int32_t *status) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t *ring = smem;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kRingBytes);
  int *prefix = reinterpret_cast<int *>(bars + kScoreWarps * kStages);
  int *nfull = prefix + batch + 1;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int gq = lane >> 2, t4 = lane & 3;  // mma groupID / thread-in-group

  // per-sequence full pages and tile counts
  for (int b = threadIdx.x; b < batch; b += blockDim.x) {
    int L = seq_lens[b];
    if (L < 0 || L > max_pages * kPage) {
      if (blockIdx.x == 0) set_status(status, LOCKS_DEV_BAD_SEQ_LEN);
      L = max(0, min(L, max_pages * kPage));
    }
    nfull[b] = L / kPage;
    prefix[b + 1] = ((L / kPage + kTilePages - 1) / kTilePages) * h_kv;
  }
  if (threadIdx.x == 0) prefix[0] = 0;
  if (lane == 0) {
    mbar_init(&bars[wid * kStages + 0], 1);
    mbar_init(&bars[wid * kStages + 1], 1);
  }
  fence_mbar_init();
  __syncthreads();
  if (wid == 0) {  // inclusive scan of prefix[1..batch]
    const int per = (batch + 31) / 32;
    const int lo = 1 + lane * per, hi = min(batch + 1, lo + per);
    int run = 0;
    for (int i = lo; i < hi; ++i) {
      run += prefix[i];
      prefix[i] = run;
    }
    int incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    const int excl = incl - run;
    for (int i = lo; i < hi; ++i) prefix[i] += excl;
  }
  __syncthreads();

  const long long total = prefix[batch];
  const long long W = (long long)gridDim.x * kScoreWarps;
  const long long gw = (long long)blockIdx.x * kScoreWarps + wid;
  const long long t_begin = gw * total / W, t_end = (gw + 1) * total / W;
  uint8_t *my_ring = ring + (size_t)wid * kStages * kTileBytes;
  uint64_t *my_bar = bars + wid * kStages;

  auto issue = [&](long long t, int stage) {
    if (lane == 0) {
      const TileInfo ti = decode_tile(t, prefix, nfull, batch, h_kv);
      const uint8_t *src =
          summaries +
          (((size_t)ti.b * h_kv + ti.h) * max_pages + ti.page0) * (size_t)kRec;
      const uint32_t bytes = (uint32_t)ti.npg * kRec;
      asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
      mbar_arrive_tx(&my_bar[stage], bytes);
      bulk_g2s(my_ring + stage * kTileBytes, src, bytes, &my_bar[stage]);
    }
  };

  if (t_begin < t_end) issue(t_begin, 0);
  if (t_begin + 1 < t_end) issue(t_begin + 1, 1);

  uint32_t qa[8][4];  // query A fragments (fp16), rows = heads of the group
  int cur_b = -1, cur_h = -1;
  bool failed = false;

  for (long long t = t_begin, it = 0; t < t_end; ++t, ++it) {
    const int stage = (int)(it & 1);
    const uint32_t phase = (uint32_t)((it >> 1) & 1);
    const TileInfo ti = decode_tile(t, prefix, nfull, batch, h_kv);
    if (!mbar_wait(&my_bar[stage], phase)) {
      failed = true;
      break;
    }
    if (ti.b != cur_b || ti.h != cur_h) {
      cur_b = ti.b;
      cur_h = ti.h;
      const __nv_bfloat16 *qb = q + ((size_t)ti.b * h_kv * G + (size_t)ti.h * G) * kDim;
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const int d0 = 16 * s + 2 * t4;
        uint32_t r0 = 0, r1 = 0, r2 = 0, r3 = 0;
        if (gq < G) {
          const uint32_t u0 = __ldg(reinterpret_cast<const uint32_t *>(qb + gq * kDim + d0));
          const uint32_t u2 = __ldg(reinterpret_cast<const uint32_t *>(qb + gq * kDim + d0 + 8));
          r0 = pack_h2(bf16_lo(u0), bf16_hi(u0));
          r2 = pack_h2(bf16_lo(u2), bf16_hi(u2));
        }
        if (WIDE && gq + 8 < G) {
          const uint32_t u1 = __ldg(reinterpret_cast<const uint32_t *>(qb + (gq + 8) * kDim + d0));
          const uint32_t u3 = __ldg(reinterpret_cast<const uint32_t *>(qb + (gq + 8) * kDim + d0 + 8));
          r1 = pack_h2(bf16_lo(u1), bf16_hi(u1));
          r3 = pack_h2(bf16_lo(u3), bf16_hi(u3));
        }
        qa[s][0] = r0;
        qa[s][1] = r1;
        qa[s][2] = r2;
        qa[s][3] = r3;
      }
    }
    const uint8_t *base = my_ring + stage * kTileBytes;

    // mma3: q . mu for the tile's 8 pages (column n = page)
    float qm[4] = {0.f, 0.f, 0.f, 0.f}, qm2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      const uint32_t u =
          gq < ti.npg ? ld_shared_u32(base + gq * kRec + kOffMu8 + 32 * t4 + 4 * s)
                      : 0u;
      if (s & 1)
        mma_f16(qm2, qa[s], i8x2_to_h2(u), i8x2_to_h2(u >> 16));
      else
        mma_f16(qm, qa[s], i8x2_to_h2(u), i8x2_to_h2(u >> 16));
    }
    float qmu0 = 0.f, qmu1 = 0.f, qmu8_0 = 0.f, qmu8_1 = 0.f;
    {
      const int p0 = 2 * t4, p1 = 2 * t4 + 1;
      const float sm0 =
          p0 < ti.npg ? __half2float(*reinterpret_cast<const __half *>(base + p0 * kRec + kOffSMu)) : 0.f;
      const float sm1 =
          p1 < ti.npg ? __half2float(*reinterpret_cast<const __half *>(base + p1 * kRec + kOffSMu)) : 0.f;
      qmu0 = (qm[0] + qm2[0]) * sm0 * kLog2eRsqrtD;
      qmu1 = (qm[1] + qm2[1]) * sm1 * kLog2eRsqrtD;
      if (WIDE) {
        qmu8_0 = (qm[2] + qm2[2]) * sm0 * kLog2eRsqrtD;
        qmu8_1 = (qm[3] + qm2[3]) * sm1 * kLog2eRsqrtD;
      }
    }

    float lse[kTilePages], lse8[kTilePages];
#pragma unroll
    for (int p = 0; p < kTilePages; ++p) {
      lse[p] = 0.f;
      lse8[p] = 0.f;
      if (p < ti.npg) {
        const uint8_t *rec = base + p * kRec;
        const uint4 vw = ld_shared_v4(rec + kOffV4 + 16 * lane);
        const uint32_t vwa[4] = {vw.x, vw.y, vw.z, vw.w};
        float a1[4] = {0.f, 0.f, 0.f, 0.f}, a1b[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const uint32_t x = vwa[w], y = x >> 8;
          mma_f16(a1, qa[2 * w], nib_lo_to_h2(x), nib_hi_to_h2(x));
          mma_f16(a1b, qa[2 * w + 1], nib_lo_to_h2(y), nib_hi_to_h2(y));
        }
        const __half2 sv = u32_as_h2(ld_shared_u32(rec + kOffSV + 4 * t4));
        const float sv0 = __low2float(sv) * kLog2eRsqrtD;
        const float sv1 = __high2float(sv) * kLog2eRsqrtD;
        const float P0 = (a1[0] + a1b[0]) * sv0, P1 = (a1[1] + a1b[1]) * sv1;
        const __half2 h01 = __floats2half2_rn(P0, P1);
        uint32_t A2[4];
        A2[0] = h2_as_u32(h01);
        A2[2] = pack_h2(P0 - __low2float(h01), P1 - __high2float(h01));
        A2[1] = 0u;
        A2[3] = 0u;
        if (WIDE) {
          const float P2 = (a1[2] + a1b[2]) * sv0, P3 = (a1[3] + a1b[3]) * sv1;
          const __half2 h23 = __floats2half2_rn(P2, P3);
          A2[1] = h2_as_u32(h23);
          A2[3] = pack_h2(P2 - __low2float(h23), P3 - __high2float(h23));
        }
        const uint32_t cw = ld_shared_u32(rec + kOffC8 + 4 * lane);
        const uint32_t bt0 = i8x2_to_h2(cw), bt1 = i8x2_to_h2(cw >> 16);
        float l0[4] = {0.f, 0.f, 0.f, 0.f}, l1[4] = {0.f, 0.f, 0.f, 0.f};
        mma_f16(l0, A2, bt0, bt0);
        mma_f16(l1, A2, bt1, bt1);
        const __half2 sc0 = u32_as_h2(ld_shared_u32(rec + kOffSC + 4 * t4));
        const __half2 sc1 = u32_as_h2(ld_shared_u32(rec + kOffSC + 16 + 4 * t4));
        const float c0 = __low2float(sc0), c1 = __high2float(sc0);
        const float c8 = __low2float(sc1), c9 = __high2float(sc1);
        lse[p] = lse2_quad(l0[0] * c0, l0[1] * c1, l1[0] * c8, l1[1] * c9);
        if (WIDE)
          lse8[p] = lse2_quad(l0[2] * c0, l0[3] * c1, l1[2] * c8, l1[3] * c9);
      }
    }
    // lane (g, t4) owns pages 2*t4 and 2*t4 + 1 of the tile
    float o0 = 0.f, o1 = 0.f, o80 = 0.f, o81 = 0.f;
#pragma unroll
    for (int p = 0; p < kTilePages; p += 2) {
      if (p == 2 * t4) {
        o0 = lse[p];
        o1 = lse[p + 1];
        o80 = lse8[p];
        o81 = lse8[p + 1];
      }
    }
    const int pg0 = 2 * t4, pg1 = 2 * t4 + 1;
    if (gq < G) {
      float *dst = s_hat + (((size_t)ti.b * h_kv + ti.h) * G + gq) * max_pages + ti.page0;
      if (pg0 < ti.npg) dst[pg0] = (o0 + qmu0) * kLn2;
      if (pg1 < ti.npg) dst[pg1] = (o1 + qmu1) * kLn2;
    }
    if (WIDE && gq + 8 < G) {
      float *dst = s_hat + (((size_t)ti.b * h_kv + ti.h) * G + gq + 8) * max_pages + ti.page0;
      if (pg0 < ti.npg) dst[pg0] = (o80 + qmu8_0) * kLn2;
      if (pg1 < ti.npg) dst[pg1] = (o81 + qmu8_1) * kLn2;
    }
    __syncwarp();
    if (t + 2 < t_end) issue(t + 2, stage);
  }
  if (failed) {
    if (lane == 0) set_status(status, LOCKS_DEV_TIMEOUT);
    // let copies still in flight land before the CTA's memory goes away
    mbar_wait(&my_bar[0], 0, 1u << 16);
    mbar_wait(&my_bar[1], 0, 1u << 16);
    mbar_wait(&my_bar[0], 1, 1u << 16);
    mbar_wait(&my_bar[1], 1, 1u << 16);
  }
}

// ---------------------------------------------------------------------------
// selection: one CTA per (sequence, KV head)
// ---------------------------------------------------------------------------
constexpr int kSelThreads = 1024;

__device__ __forceinline__ uint32_t order_key(float x) {
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
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
    int wa = sh[lane], wb = sh[32 + lane];
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

__global__ void __launch_bounds__(kSelThreads)
    select_kernel(const float *__restrict__ scores,
                  const int32_t *__restrict__ seq_lens, int h_kv, int G,
                  int max_pages, int k, int32_t *__restrict__ idx,
                  uint32_t *__restrict__ keybuf, int32_t *status) {
  __shared__ float zs[kMaxGroup];
  __shared__ float red_m[32][kMaxGroup], red_s[32][kMaxGroup];
  __shared__ int hist[256];
  __shared__ int sh_scan[64];
  __shared__ uint32_t sh_prefix, sh_mask;
  __shared__ int sh_remaining;

  const int b = blockIdx.y, h = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  int L = seq_lens[b];
  if (L < 0 || L > max_pages * kPage) {
    if (tid == 0 && h == 0) set_status(status, LOCKS_DEV_BAD_SEQ_LEN);
    L = max(0, min(L, max_pages * kPage));
  }
  const int n = (L + kPage - 1) / kPage, nf = L / kPage;
  int32_t *out = idx + ((size_t)b * h_kv + h) * k;
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
  uint32_t *keys = keybuf + ((size_t)b * h_kv + h) * (size_t)max_pages;

  // Z_g: log-sum-exp over all summarised pages (base-2 units)
  constexpr float kLog2e = 1.4426950408889634f;
  for (int g = 0; g < G; ++g) {
    float m = -INFINITY, s = 0.f;
    for (int j = tid; j < nf; j += blockDim.x) {
      const float x = sc[(size_t)g * max_pages + j] * kLog2e;
      if (x > m) {
        s = s * exp2f(m - x) + 1.f;
        m = x;
      } else {
        s += exp2f(x - m);
      }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
      const float mm = fmaxf(m, m2);
      s = (m == -INFINITY ? 0.f : s * exp2f(m - mm)) +
          (m2 == -INFINITY ? 0.f : s2 * exp2f(m2 - mm));
      m = mm;
    }
    if (lane == 0) {
      red_m[wid][g] = m;
      red_s[wid][g] = s;
    }
  }
  __syncthreads();
  if (tid < G) {
    float m = -INFINITY;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) m = fmaxf(m, red_m[w][tid]);
    float s = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w)
      if (red_m[w][tid] != -INFINITY) s += red_s[w][tid] * exp2f(red_m[w][tid] - m);
    zs[tid] = m + log2f(s);
  }
  __syncthreads();

  // share-average key per candidate page j in [1, n-2]:
  // log2 of sum_g 2^(s_gj - Z_g) (the constant log2 G dropped)
  const int ncand = n - 2;
  for (int c = tid; c < ncand; c += blockDim.x) {
    const int j = c + 1;
    float m = -INFINITY;
    for (int g = 0; g < G; ++g)
      m = fmaxf(m, sc[(size_t)g * max_pages + j] * kLog2e - zs[g]);
    float s = 0.f;
    for (int g = 0; g < G; ++g)
      s += exp2f(sc[(size_t)g * max_pages + j] * kLog2e - zs[g] - m);
    keys[c] = order_key(m + log2f(s));
  }
  if (tid == 0) {
    sh_prefix = 0u;
    sh_mask = 0u;
    sh_remaining = k - 2;
  }
  __syncthreads();

  // radix select of the (k-2)-th largest key, 8-bit digits, MSB first
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    const uint32_t pre = sh_prefix, msk = sh_mask;
    for (int c = tid; c < ncand; c += blockDim.x) {
      const uint32_t u = keys[c];
      if ((u & msk) == pre) atomicAdd(&hist[(u >> shift) & 255u], 1);
    }
    __syncthreads();
    if (wid == 0) {
      // lane l covers digits 255-8l .. 248-8l (descending)
      int cnt[8], tot = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        cnt[i] = hist[255 - 8 * lane - i];
        tot += cnt[i];
      }
      int incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      const int before = incl - tot;
      const int rem = sh_remaining;
      if (before < rem && rem <= incl) {
        int acc = before;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (acc < rem && rem <= acc + cnt[i]) {
            sh_prefix = pre | ((uint32_t)(255 - 8 * lane - i) << shift);
            sh_mask = msk | (255u << shift);
            sh_remaining = rem - acc;
          }
          acc += cnt[i];
        }
      }
    }
    __syncthreads();
  }
  const uint32_t T = sh_prefix;
  const int need_eq = sh_remaining;  // keys equal to T to keep (lowest j)

  // ordered compaction over contiguous chunks of candidates
  const int chunk = (ncand + blockDim.x - 1) / blockDim.x;
  const int lo = min(ncand, tid * chunk), hi = min(ncand, lo + chunk);
  int gt = 0, eq = 0;
  for (int c = lo; c < hi; ++c) {
    const uint32_t u = keys[c];
    gt += u > T;
    eq += u == T;
  }
  int gt_before, eq_before;
  block_scan2(gt, eq, gt_before, eq_before, sh_scan);
  int g_loc = 0, e_loc = 0;
  for (int c = lo; c < hi; ++c) {
    const uint32_t u = keys[c];
    bool sel = false;
    if (u > T) {
      sel = true;
    } else if (u == T && eq_before + e_loc < need_eq) {
      sel = true;
    }
    if (sel) {
      const int pos = 1 + gt_before + g_loc + min(eq_before + e_loc, need_eq);
      if (pos >= 1 && pos < k - 1)
        out[pos] = c + 1;
      else
        set_status(status, LOCKS_DEV_BAD_INDEX);
    }
    g_loc += u > T;
    e_loc += u == T;
  }
  if (tid == 0) {
    out[0] = 0;
    out[k - 1] = n - 1;
  }
}

// --------------------------------------------------------------------------
// launchers
// --------------------------------------------------------------------------
static int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

size_t score_smem_bytes(int batch) {
  return (size_t)kRingBytes + sizeof(uint64_t) * kScoreWarps * kStages +
         sizeof(int) * (2 * (size_t)batch + 1);
}

int score_max_batch() {
  // the per-sequence tables must fit next to the ring in 227 KB
  return (int)((227 * 1024 - (size_t)kRingBytes -
                sizeof(uint64_t) * kScoreWarps * kStages - 64) /
               (2 * sizeof(int)));
}

cudaError_t launch_score(const void *q, const void *summaries,
                         const int32_t *seq_lens, int batch, int h_kv, int G,
                         int max_pages, float *s_hat, int32_t *status,
                         cudaStream_t stream) {
  const size_t smem = score_smem_bytes(batch);
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(
        score_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
        227 * 1024);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(score_kernel<true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             227 * 1024);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int grid = sm_count();
  if (G > 8)
    score_kernel<true><<<grid, kScoreThreads, smem, stream>>>(
        static_cast<const __nv_bfloat16 *>(q),
        static_cast<const uint8_t *>(summaries), seq_lens, batch, h_kv, G,
        max_pages, s_hat, status);
  else
    score_kernel<false><<<grid, kScoreThreads, smem, stream>>>(
        static_cast<const __nv_bfloat16 *>(q),
        static_cast<const uint8_t *>(summaries), seq_lens, batch, h_kv, G,
        max_pages, s_hat, status);
  return cudaGetLastError();
}

cudaError_t launch_select(const float *scores, const int32_t *seq_lens,
                          int batch, int h_kv, int G, int max_pages, int k,
                          int32_t *idx, uint32_t *keybuf, int32_t *status,
                          cudaStream_t stream) {
  dim3 grid(h_kv, batch);
  select_kernel<<<grid, kSelThreads, 0, stream>>>(
      scores, seq_lens, h_kv, G, max_pages, k, idx, keybuf, status);
  return cudaGetLastError();
}

}  // namespace locks
