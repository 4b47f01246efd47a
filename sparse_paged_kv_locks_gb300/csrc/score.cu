// Summary scoring (LOCKS reading notes §4.2 Eq.(4), §4.4 Algorithm 2).
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
#include "score_ops.cuh"
#include "select_top.cuh"

namespace locks {

constexpr int kScoreWarps = 16;
constexpr int kScoreThreads = 32 * kScoreWarps;
constexpr int kTilePages = 8;
constexpr int kTileBytes = kTilePages * kRec;  // 6656
constexpr int kStages = 2;
constexpr int kRingBytes = kScoreWarps * kStages * kTileBytes;

// The basis and coefficient products and the per-page log-sum-exp for the
// pages of one tile, two pages per step (G <= 8).  Product 1 is transposed:
// rows 0..7 are page A's basis components, rows 8..15 page B's (A operand =
// unpacked codes, straight into the fragment registers), columns are query
// heads (B operand = the query, resident).  The 8x8 (component x head)
// blocks are turned with movmatrix into head-major operands for product 2.
// Lane (gq, t4) keeps the value of pair t4.  SAFE selects the max-subtracted
// log-sum-exp; otherwise the return value folds every quad sum's distance
// from the normal range (>= kLseBad: recompute with SAFE).
template <int MODE, bool SAFE>
__device__ __forceinline__ uint32_t score_pairs(
    uint32_t base_s, int npg, int lane, const uint32_t (&qv)[8][2],
    float offc0, float offc1, float vscale, float &keepA, float &keepB) {
  const int gq = lane >> 2, t4 = lane & 3;
  const bool lowh = gq < 4;
  const uint32_t maskA = lowh ? 0xffffffffu : 0u;
  uint32_t bad = 0u;
#pragma unroll 1
  for (int pp = 0; 2 * pp < npg; ++pp) {
    const uint32_t ra = base_s + (uint32_t)(2 * pp) * kRec;
    const uint32_t rb = ra + kRec;
    const uint4 va = lds128(ra + kOffV4 + 16 * lane);
    const uint4 vb = lds128(rb + kOffV4 + 16 * lane);
    const uint32_t ca = lds32(ra + kOffC8 + 4 * lane);
    const uint32_t cb = lds32(rb + kOffC8 + 4 * lane);
    // sV of component gq in each page
    const uint32_t svo = kOffSV + 16 * (gq >> 1) + 2 * (gq & 1);
    const float sva = __half2float(__ushort_as_half(
                          (unsigned short)lds16(ra + svo))) * vscale;
    const float svb = __half2float(__ushort_as_half(
                          (unsigned short)lds16(rb + svo))) * vscale;
    const uint32_t vaw[4] = {va.x, va.y, va.z, va.w};
    const uint32_t vbw[4] = {vb.x, vb.y, vb.z, vb.w};
    float d0[4], d1[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const uint32_t xa = vaw[w], xb = vbw[w];
      const uint32_t za = xa >> 8, zb = xb >> 8;
      const uint32_t a0[4] = {nib_f16_lo(xa), nib_f16_lo(xb),
                              nib_f16_hi(xa), nib_f16_hi(xb)};
      const uint32_t a1[4] = {nib_f16_lo(za), nib_f16_lo(zb),
                              nib_f16_hi(za), nib_f16_hi(zb)};
      if (w == 0) {
        mma_f16_c(d0, a0, qv[0][0], qv[0][1], offc0, offc1, offc0,
                  offc1);
        mma_f16_c(d1, a1, qv[1][0], qv[1][1], 0.f, 0.f, 0.f, 0.f);
      } else {
        mma_f16(d0, a0, qv[2 * w][0], qv[2 * w][1]);
        mma_f16(d1, a1, qv[2 * w + 1][0], qv[2 * w + 1][1]);
      }
    }
    // proj (log2 units) = D * sV * log2(e)/sqrt(d), split hi + lo fp16
    const float pa0 = (d0[0] + d1[0]) * sva, pa1 = (d0[1] + d1[1]) * sva;
    const float pb0 = (d0[2] + d1[2]) * svb, pb1 = (d0[3] + d1[3]) * svb;
    const __half2 ha = __floats2half2_rn(pa0, pa1);
    const __half2 hb = __floats2half2_rn(pb0, pb1);
    const uint32_t la = split_lo(h2_as_u32(ha), pa0, pa1);
    const uint32_t lb = split_lo(h2_as_u32(hb), pb0, pb1);
    const uint32_t tha = movmatrix_trans(h2_as_u32(ha));
    const uint32_t tla = movmatrix_trans(la);
    const uint32_t thb = movmatrix_trans(h2_as_u32(hb));
    const uint32_t tlb = movmatrix_trans(lb);
    uint32_t ba0, ba1, bb0, bb1;
    i8x4_to_h2(ca, ba0, ba1);
    i8x4_to_h2(cb, bb0, bb1);
    float l0[4], l1[4];
    if constexpr (MODE == 1) {
      // rows 0-3: page A heads (high halves, k 0..7 = page A comps),
      // rows 4-7: page B heads (high, k 8..15 = page B comps),
      // rows 8-15: the same with the low halves
      const uint32_t A2[4] = {tha & maskA, tla & maskA, thb & ~maskA,
                              tlb & ~maskA};
      mma_f16_z(l0, A2, ba0, bb0);
      mma_f16_z(l1, A2, ba1, bb1);
      const uint32_t rs = lowh ? ra : rb;
      const uint4 sc = lds128(rs + kOffSV + 16 * t4);
      const __half2 s0 = u32_as_h2(sc.y), s1 = u32_as_h2(sc.z);
      const float e = lse2_quad_sel((l0[0] + l0[2]) * __low2float(s0),
                                    (l0[1] + l0[3]) * __high2float(s0),
                                    (l1[0] + l1[2]) * __low2float(s1),
                                    (l1[1] + l1[3]) * __high2float(s1),
                                    SAFE, bad);
      if (pp == t4) keepA = e;
    } else {
      float m0[4], m1[4];
      mma1688_f16_z(l0, tha, tla, ba0);
      mma1688_f16_z(l1, tha, tla, ba1);
      mma1688_f16_z(m0, thb, tlb, bb0);
      mma1688_f16_z(m1, thb, tlb, bb1);
      const uint4 sa = lds128(ra + kOffSV + 16 * t4);
      const uint4 sb = lds128(rb + kOffSV + 16 * t4);
      const __half2 a0 = u32_as_h2(sa.y), a1 = u32_as_h2(sa.z);
      const __half2 b0 = u32_as_h2(sb.y), b1 = u32_as_h2(sb.z);
      const float ea = lse2_quad_sel((l0[0] + l0[2]) * __low2float(a0),
                                     (l0[1] + l0[3]) * __high2float(a0),
                                     (l1[0] + l1[2]) * __low2float(a1),
                                     (l1[1] + l1[3]) * __high2float(a1),
                                     SAFE, bad);
      const float eb = lse2_quad_sel((m0[0] + m0[2]) * __low2float(b0),
                                     (m0[1] + m0[3]) * __high2float(b0),
                                     (m1[0] + m1[2]) * __low2float(b1),
                                     (m1[1] + m1[3]) * __high2float(b1),
                                     SAFE, bad);
      if (pp == t4) {
        keepA = ea;
        keepB = eb;
      }
    }
  }
  return bad;
}


// lane 0 starts the bulk copy of tile c into `dst`, completing on `bar`
__device__ __forceinline__ void issue_tile(const Cursor &c, const int *nfull,
                                           const uint8_t *summaries, int h_kv,
                                           int max_pages, uint8_t *dst,
                                           uint64_t *bar, int lane) {
  if (lane == 0) {
    const int page0 = c.j * kTilePages;
    const int npg = min(kTilePages, nfull[c.b] - page0);
    const uint8_t *src =
        summaries +
        (((size_t)c.b * h_kv + c.h) * max_pages + page0) * (size_t)kRec;
    const uint32_t bytes = (uint32_t)npg * kRec;
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
    mbar_arrive_tx(bar, bytes);
    bulk_g2s(dst, src, bytes, bar);
  }
}

// Running sums of 2^v (v in log2 units) as (reference r, sum s of
// 2^(v - r)): r is raised, and s rescaled, only when v passes it by more
// than 2^6, so every term stays below 2^64.  A NaN makes r = +inf.
__device__ __forceinline__ void norm_add(float &r, float &s, float v) {
  if (!(v > -INFINITY)) {  // -inf adds nothing
    if (v != v) r = INFINITY;
    return;
  }
  if (v > r + 64.f) {  // also the first value (r = -inf)
    s = r == -INFINITY ? 0.f : s * ex2_fast(r - v);
    r = v;
  }
  s += ex2_fast(v - r);
}

// (r, s) <- (r, s) + (r2, s2) in the same sense
__device__ __forceinline__ void norm_merge(float &r, float &s, float r2,
                                           float s2) {
  const float m = fmaxf(r, r2);
  if (m == -INFINITY) return;
  s = (r == -INFINITY ? 0.f : s * ex2_fast(r - m)) +
      (r2 == -INFINITY ? 0.f : s2 * ex2_fast(r2 - m));
  r = m;
}

__device__ __forceinline__ void norm_merge_xor(float &r, float &s, int o) {
  const float r2 = __shfl_xor_sync(0xffffffffu, r, o);
  const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
  norm_merge(r, s, r2, s2);
}

// Longest page list the fused form takes: its CTA 0 keeps the unit's keys
// and the radix scratch in the (by then idle) tile ring.
constexpr int kFusedMaxPages = 8192;
static_assert(kFusedMaxPages * 4 + sizeof(SelectScratch) + 16 <= kRingBytes,
              "fused keys and scratch must fit the tile ring");

// The selection of the fused form, after the cluster's warps scored unit
// (b, h) into s_hat.  (nr, ns): this lane's running pair of its head
// (MODE 1: gq & 3, else gq).  Every thread of every CTA of the cluster
// calls it.
template <int MODE>
__device__ __forceinline__ void fused_select_epilogue(
    float nr, float ns, const float *s_hat, const int32_t *seq_lens,
    int h_kv, int G, int max_pages, int k, int b, int h, int rank, int csize,
    int tiles, uint8_t *smem, int32_t *idx_out, int32_t *status) {
  __shared__ float f_r[kScoreWarps][kMaxGroup], f_s[kScoreWarps][kMaxGroup];
  __shared__ float f_pr[kMaxGroup], f_ps[kMaxGroup], f_z[kMaxGroup];
  __shared__ uint32_t f_red[2][kScoreWarps];
  __shared__ uint32_t f_kmm[2][8];  // CTA 0: (kmin, kmax) of every rank
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int gq = lane >> 2, t4 = lane & 3;
  // this CTA's pair per head: lanes of a head, then warps
  norm_merge_xor(nr, ns, 1);
  norm_merge_xor(nr, ns, 2);
  if (MODE == 1) norm_merge_xor(nr, ns, 16);
  if (t4 == 0 && (MODE != 1 || gq < 4) && gq < G) {
    f_r[wid][gq] = nr;
    f_s[wid][gq] = ns;
  }
  __syncthreads();
  if (tid < G) {
    float r = -INFINITY, sm = 0.f;
    for (int w = 0; w < kScoreWarps; ++w) norm_merge(r, sm, f_r[w][tid], f_s[w][tid]);
    f_pr[tid] = r;
    f_ps[tid] = sm;
  }
  cluster_sync();  // every CTA scored its pages and holds its pairs
  // Z_g (log2 units): the cluster's pairs merged in rank order, the same
  // value in every CTA
  if (tid < G) {
    float r = -INFINITY, sm = 0.f;
    for (int c = 0; c < csize; ++c)
      norm_merge(r, sm, ld_cluster_f32(mapa_shared(smem_u32(&f_pr[tid]), c)),
                 ld_cluster_f32(mapa_shared(smem_u32(&f_ps[tid]), c)));
    f_z[tid] = r + lg2_fast(sm);
  }
  int L = seq_lens[b];
  L = max(0, min(L, max_pages * kPage));
  const int n = (L + kPage - 1) / kPage, nf = L / kPage;
  // CTA 0's tile ring, idle now: keys of the unit's pages, then the radix
  // scratch
  uint32_t *keys = reinterpret_cast<uint32_t *>(smem);
  SelectScratch &sel = *reinterpret_cast<SelectScratch *>(
      smem + ((size_t)max_pages * 4 + 15) / 16 * 16);
  const uint32_t keys_s = smem_u32(keys);
  if (rank == 0) {
    for (int j = nf + tid; j < n; j += blockDim.x) keys[j] = 0u;
    for (int i = tid; i < kRadixBins; i += blockDim.x) sel.hist[0][i] = 0;
  }
  __syncthreads();
  // keys of this CTA's full pages (the tiles its warps scored):
  // log2 sum_g 2^(s_gj - Z_g), the share-average up to the factor 1/G
  const long long nwc = (long long)csize * kScoreWarps;
  const int p0 = (int)((long long)rank * kScoreWarps * tiles / nwc) *
                 kTilePages;
  const int p1 = min(nf, (int)((long long)(rank + 1) * kScoreWarps * tiles /
                               nwc) * kTilePages);
  const float *sc = s_hat + ((size_t)b * h_kv + h) * G * (size_t)max_pages;
  constexpr float kLog2e = 1.4426950408889634f;
  uint32_t kmin = 0xffffffffu, kmax = 0u;
  for (int j = p0 + tid; j < p1; j += blockDim.x) {
    float sum = 0.f, m = -INFINITY;
    for (int g = 0; g < G; ++g) {
      const float x = fmaf(sc[(size_t)g * max_pages + j], kLog2e, -f_z[g]);
      sum += ex2_fast(x);
      m = fmaxf(m, x);
    }
    float key = lg2_fast(sum);
    if (!(sum > 0.f && sum < INFINITY)) {  // every term underflowed
      float t = 0.f;
      for (int g = 0; g < G; ++g)
        t += ex2_fast(fmaf(sc[(size_t)g * max_pages + j], kLog2e, -f_z[g]) -
                      m);
      key = m + lg2_fast(t);
    }
    const bool cand = (unsigned)(j - 1) <= (unsigned)(n - 3);
    const uint32_t kq = cand ? order_key(key) : 0u;
    st_cluster_u32(mapa_shared(keys_s + 4u * (uint32_t)j, 0), kq);
    if (cand) {
      kmin = min(kmin, kq);
      kmax = max(kmax, kq);
    }
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
    kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
  }
  if (lane == 0) {
    f_red[0][wid] = kmin;
    f_red[1][wid] = kmax;
  }
  __syncthreads();
  if (tid == 0) {
    for (int w = 1; w < kScoreWarps; ++w) {
      kmin = min(kmin, f_red[0][w]);
      kmax = max(kmax, f_red[1][w]);
    }
    st_cluster_u32(mapa_shared(smem_u32(&f_kmm[0][rank]), 0), kmin);
    st_cluster_u32(mapa_shared(smem_u32(&f_kmm[1][rank]), 0), kmax);
  }
  cluster_sync();  // CTA 0 holds every key and every rank's bounds
  if (rank != 0) return;
  int32_t *out = idx_out + ((size_t)b * h_kv + h) * k;
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
  uint32_t a = 0xffffffffu, z = 0u;
  if (tid == 0)
    for (int c = 0; c < csize; ++c) {
      a = min(a, f_kmm[0][c]);
      z = max(z, f_kmm[1][c]);
    }
  select_top<true, kScoreWarps>(keys, true, n, k, a, z, out, status, sel);
}

// FUSED: the single-launch score-and-select form for short page lists.
// The grid is one cluster of C CTAs per (sequence, KV head) unit; the C x
// 16 warps of a cluster split that unit's tiles, and after scoring the
// cluster forms the mass-fraction denominators from per-CTA partial sums
// (distributed shared memory), each CTA computes its pages' selection keys
// into CTA 0's shared memory, and CTA 0 selects (select_top) into idx_out.
template <int MODE, bool FUSED = false>
__global__ void __launch_bounds__(kScoreThreads, 1)
    score_kernel(const __nv_bfloat16 *__restrict__ q,
                 const uint8_t *__restrict__ summaries,
                 const int32_t *__restrict__ seq_lens, int batch, int h_kv,
                 int G, int max_pages, float *__restrict__ s_hat,
                 int32_t *status, int wait_query, int k,
                 int32_t *__restrict__ idx_out) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t *ring = smem;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kRingBytes);
  int *prefix = reinterpret_cast<int *>(bars + kScoreWarps * kStages);
  int *nfull = prefix + batch + 1;
  int *tph = nfull + batch;  // tiles per KV head of each sequence
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int gq = lane >> 2, t4 = lane & 3;  // mma groupID / thread-in-group
  // selection may launch now; it waits for these scores before reading them
  pdl_trigger();
  const uint64_t keep = l2_keep_policy();

  // per-sequence full pages and tile counts
  for (int b = threadIdx.x; b < batch; b += blockDim.x) {
    int L = seq_lens[b];
    if (L < 0 || L > max_pages * kPage) {
      if (blockIdx.x == 0) set_status(status, LOCKS_DEV_BAD_SEQ_LEN);
      L = max(0, min(L, max_pages * kPage));
    }
    nfull[b] = L / kPage;
    tph[b] = (L / kPage + kTilePages - 1) / kTilePages;
    prefix[b + 1] = tph[b] * h_kv;
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

  long long t_begin, t_end;
  int fu_b = 0, fu_h = 0, fu_rank = 0, fu_size = 1;  // FUSED: the unit
  if constexpr (FUSED) {
    fu_rank = (int)cluster_ctarank();
    fu_size = (int)cluster_nctarank();
    const int u = (int)(blockIdx.x / fu_size);
    fu_b = u / h_kv;
    fu_h = u - fu_b * h_kv;
    const long long t0 = prefix[fu_b] + (long long)fu_h * tph[fu_b];
    const long long nt = tph[fu_b];
    const long long lw = (long long)fu_rank * kScoreWarps + wid;
    const long long nw = (long long)fu_size * kScoreWarps;
    t_begin = t0 + lw * nt / nw;
    t_end = t0 + (lw + 1) * nt / nw;
  } else {
    const long long total = prefix[batch];
    const long long W = (long long)gridDim.x * kScoreWarps;
    const long long gw = (long long)blockIdx.x * kScoreWarps + wid;
    t_begin = gw * total / W;
    t_end = (gw + 1) * total / W;
    // wait_query: the query comes from the preceding kernel (this one is
    // its programmatic dependent), so every thread waits for it before
    // reading q or exiting.
    if (t_begin >= t_end) {
      if (wait_query) pdl_wait();
      return;
    }
  }
  uint8_t *my_ring = ring + (size_t)wid * kStages * kTileBytes;
  const uint32_t ring_s = smem_u32(my_ring);
  uint64_t *my_bar = bars + wid * kStages;

  Cursor cur{0, 0, 0};
  Cursor nxt = cur;
  if (t_begin < t_end) {
    {  // largest b with prefix[b] <= t_begin
      int lo = 0, hi = batch;
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (prefix[mid] <= t_begin) lo = mid; else hi = mid;
      }
      const int rem = (int)(t_begin - prefix[lo]);
      const int tb = tph[lo];
      cur.b = lo;
      cur.h = rem / tb;
      cur.j = rem - cur.h * tb;
    }
    nxt = cur;
    issue_tile(nxt, nfull, summaries, h_kv, max_pages, my_ring, &my_bar[0],
               lane);
    advance_cursor(nxt, tph, batch, h_kv);
    if (t_begin + 1 < t_end) {
      issue_tile(nxt, nfull, summaries, h_kv, max_pages, my_ring + kTileBytes,
                 &my_bar[1], lane);
      advance_cursor(nxt, tph, batch, h_kv);
    }
  }
  if (wait_query) pdl_wait();  // first two tiles in flight; q is read next

  constexpr bool WIDE = MODE == 3;
  uint32_t qb[8][4];  // query A fragments, bf16 (basis product, one page)
  uint32_t qh[8][4];  // query A fragments, fp16 (centroid product)
  uint32_t qv[8][2];  // query B fragments, fp16 (basis product, two pages;
                      // k 8..15 of each step hold q / 16)
  float offc0 = 0.f, offc1 = 0.f;  // offsets of columns 2*t4, 2*t4 + 1
  float off_v = 0.f, off_v8 = 0.f, off_m = 0.f, off_m8 = 0.f;
  // fp16 operands carry the query times 2^-e (e > 0 only when some |q| of
  // the unit reaches 2^14); these undo it in log2 units
  float vscale = kLog2eRsqrtD, mscale = kLog2eRsqrtD;
  int cur_b = -1, cur_h = -1;
  bool failed = false;
  // this lane's score rows of the current unit (MODE 3: heads gq, gq + 8;
  // MODE 1: head gq & 3; MODE 2: head gq)
  float *lane_row = nullptr, *lane_row8 = nullptr;
  const int n_tiles = (int)(t_end - t_begin);
  // FUSED: this lane's running (reference, sum of 2^(v - reference)) over
  // the scores it writes (log2 units), for head gq & 3 (MODE 1) or gq
  float nr = -INFINITY, ns = 0.f;

  for (int it = 0; it < n_tiles; ++it) {
    const int stage = it & 1;
    const uint32_t phase = (uint32_t)((it >> 1) & 1);
    if (cur.b != cur_b || cur.h != cur_h) {
      cur_b = cur.b;
      cur_h = cur.h;
      float *unit_rows =
          s_hat + ((size_t)cur.b * h_kv + cur.h) * G * (size_t)max_pages;
      lane_row = unit_rows + (size_t)(MODE == 1 ? (gq & 3) : gq) * max_pages;
      lane_row8 = unit_rows + (size_t)(gq + 8) * max_pages;
      const __nv_bfloat16 *qrow =
          q + ((size_t)cur.b * h_kv * G + (size_t)cur.h * G) * kDim;
      float amax = 0.f;
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const int d0 = 16 * s + 2 * t4;
        uint32_t u0 = 0, u2 = 0, u1 = 0, u3 = 0;
        if (gq < G) {
          u0 = __ldg(reinterpret_cast<const uint32_t *>(qrow + gq * kDim + d0));
          u2 = __ldg(reinterpret_cast<const uint32_t *>(qrow + gq * kDim + d0 + 8));
        }
        if (WIDE && gq + 8 < G) {
          u1 = __ldg(reinterpret_cast<const uint32_t *>(qrow + (gq + 8) * kDim + d0));
          u3 = __ldg(reinterpret_cast<const uint32_t *>(qrow + (gq + 8) * kDim + d0 + 8));
        }
        qb[s][0] = u0;
        qb[s][1] = u1;
        qb[s][2] = u2;
        qb[s][3] = u3;
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(bf16_lo(u0)), fabsf(bf16_hi(u0))),
                                 fmaxf(fabsf(bf16_lo(u2)), fabsf(bf16_hi(u2)))));
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(bf16_lo(u1)), fabsf(bf16_hi(u1))),
                                 fmaxf(fabsf(bf16_lo(u3)), fabsf(bf16_hi(u3)))));
      }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      // power-of-two prescale keeping every fp16 operand below 2^14
      const int ex =
          amax >= 16384.f ? ((__float_as_int(amax) >> 23) & 0xff) - 140 : 0;
      const float qsc = __int_as_float((127 - ex) << 23);  // 2^-ex
      const float qun = __int_as_float((127 + ex) << 23);  // 2^ex
      mscale = kLog2eRsqrtD * qun;
      vscale = MODE == 3 ? kLog2eRsqrtD : kLog2eRsqrtD * qun;
      float sum = 0.f, sum8 = 0.f, sumh = 0.f, sumh8 = 0.f;
#pragma unroll
      for (int s = 0; s < 8; ++s) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t u = qb[s][i];
          const __half2 hq =
              __floats2half2_rn(bf16_lo(u) * qsc, bf16_hi(u) * qsc);
          qh[s][i] = h2_as_u32(hq);
          const float bs = bf16_lo(u) + bf16_hi(u);
          const float hs = __low2float(hq) + __high2float(hq);
          if (i & 1) {
            sum8 += bs;
            sumh8 += hs;
          } else {
            sum += bs;
            sumh += hs;
          }
        }
      }
#pragma unroll
      for (int o = 1; o <= 2; o <<= 1) {
        sum += __shfl_xor_sync(0xffffffffu, sum, o);
        sum8 += __shfl_xor_sync(0xffffffffu, sum8, o);
        sumh += __shfl_xor_sync(0xffffffffu, sumh, o);
        sumh8 += __shfl_xor_sync(0xffffffffu, sumh8, o);
      }
      if constexpr (MODE != 3) {
        // column n of the transposed basis product is query head
        // (n mod 4) for G <= 4 and head n for G <= 8
        const int hc = MODE == 1 ? (gq & 3) : gq;
        const __nv_bfloat16 *qc = qrow + hc * kDim;
        float clo = 0.f, chi = 0.f;
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          const int d0 = 16 * s + 2 * t4;
          const uint32_t u =
              hc < G ? __ldg(reinterpret_cast<const uint32_t *>(qc + d0)) : 0u;
          const uint32_t u8 =
              hc < G ? __ldg(reinterpret_cast<const uint32_t *>(qc + d0 + 8))
                     : 0u;
          const __half2 lo =
              __floats2half2_rn(bf16_lo(u) * qsc, bf16_hi(u) * qsc);
          const __half2 hi = __floats2half2_rn(bf16_lo(u8) * qsc * 0.0625f,
                                               bf16_hi(u8) * qsc * 0.0625f);
          qv[s][0] = h2_as_u32(lo);
          qv[s][1] = h2_as_u32(hi);
          clo += __low2float(lo) + __high2float(lo);
          chi += __low2float(hi) + __high2float(hi);
        }
        // cancels the 1032 (k 0..7) and 1152 (k 8..15) of every basis code
        float cs = -1032.f * clo - 1152.f * chi;
        cs += __shfl_xor_sync(0xffffffffu, cs, 1);
        cs += __shfl_xor_sync(0xffffffffu, cs, 2);
        // offsets of columns 2*t4 and 2*t4 + 1
        offc0 = __shfl_sync(0xffffffffu, cs, 4 * (2 * t4));
        offc1 = __shfl_sync(0xffffffffu, cs, 4 * (2 * t4 + 1));
      }
      off_v = -136.f * sum;     // cancels the +136 of every bf16 basis code
      off_v8 = -136.f * sum8;
      off_m = -1152.f * sumh;   // cancels the +1152 of every centroid code
      off_m8 = -1152.f * sumh8;
    }
    const int page0 = cur.j * kTilePages;
    const int npg = min(kTilePages, nfull[cur.b] - page0);
    if (!mbar_wait(&my_bar[stage], phase)) {
      failed = true;
      break;
    }
    const uint32_t base_s = ring_s + stage * kTileBytes;
    if constexpr (MODE != 3) {
      // An odd page count leaves the second page of the last pair unused:
      // its slot is zeroed (a zero record scores to a finite constant) so
      // that what the ring held before cannot take part in the overflow
      // vote below and change how the tile's pages are computed.
      if (npg & 1) {
        uint4 *slot = reinterpret_cast<uint4 *>(my_ring + stage * kTileBytes +
                                                npg * kRec);
        for (int i = lane; i < kRec / 16; i += 32)
          slot[i] = make_uint4(0u, 0u, 0u, 0u);
        __syncwarp();
      }
      float keepA = 0.f, keepB = 0.f;
      // first pass without per-pair overflow checks; a second, max-
      // subtracted pass only when some quad sum left the normal range
      const uint32_t bad = score_pairs<MODE, false>(
          base_s, npg, lane, qv, offc0, offc1, vscale, keepA, keepB);
      if (__any_sync(0xffffffffu, bad >= kLseBad))
        score_pairs<MODE, true>(base_s, npg, lane, qv, offc0, offc1, vscale,
                                keepA, keepB);
      // q . mu for the tile's 8 pages (column n = page gq of the tile)
      float qm[4] = {off_m, off_m, off_m8, off_m8};
      float qm2[4] = {0.f, 0.f, 0.f, 0.f};
      {
        const uint32_t mrow = base_s + gq * kRec + kOffMu8 + 32 * t4;
        const uint4 m0 = lds128(mrow), m1 = lds128(mrow + 16);
        const uint32_t mw[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          uint32_t b01, b23;
          i8x4_to_h2_off(mw[s], b01, b23);
          if (s & 1)
            mma_f16(qm2, qh[s], b01, b23);
          else
            mma_f16(qm, qh[s], b01, b23);
        }
      }
      const float qm_lo = qm[0] + qm2[0], qm_hi = qm[1] + qm2[1];
      if constexpr (MODE == 1) {
        // lane (g, t4) of the low half owns page 2*t4, of the high half page
        // 2*t4 + 1, head g & 3
        const bool up = lane >= 16;
        const float qm_from_low = __shfl_xor_sync(0xffffffffu, qm_hi, 16);
        const int pg = 2 * t4 + (up ? 1 : 0);
        const int head = gq & 3;
        const float smu = __half2float(__ushort_as_half(
            (unsigned short)lds16(base_s + pg * kRec + kOffSMu)));
        const float qmu = up ? qm_from_low : qm_lo;
        if (head < G && pg < npg) {
          const float v = keepA + qmu * smu * mscale;  // log2 units
          st_keep(lane_row + page0 + pg, v * kLn2, keep);
          if constexpr (FUSED) norm_add(nr, ns, v);
        }
      } else {
        const int pg0 = 2 * t4, pg1 = pg0 + 1;
        const float sm0 = __half2float(__ushort_as_half(
            (unsigned short)lds16(base_s + pg0 * kRec + kOffSMu)));
        const float sm1 = __half2float(__ushort_as_half(
            (unsigned short)lds16(base_s + pg1 * kRec + kOffSMu)));
        if (gq < G) {
          if (pg0 < npg) {
            const float v = keepA + qm_lo * sm0 * mscale;
            st_keep(lane_row + page0 + pg0, v * kLn2, keep);
            if constexpr (FUSED) norm_add(nr, ns, v);
          }
          if (pg1 < npg) {
            const float v = keepB + qm_hi * sm1 * mscale;
            st_keep(lane_row + page0 + pg1, v * kLn2, keep);
            if constexpr (FUSED) norm_add(nr, ns, v);
          }
        }
      }
    } else {
      // one page per mma group, heads in all 16 rows
      float o0 = 0.f, o1 = 0.f, o80 = 0.f, o81 = 0.f;
#pragma unroll
      for (int p = 0; p < kTilePages; ++p) {
        if (p < npg) {
          const uint32_t rec = base_s + p * kRec;
          const uint4 vw = lds128(rec + kOffV4 + 16 * lane);
          const uint4 sc = lds128(rec + kOffSV + 16 * t4);
          const uint32_t cw = lds32(rec + kOffC8 + 4 * lane);
          const uint32_t vwa[4] = {vw.x, vw.y, vw.z, vw.w};
          float a1[4] = {off_v, off_v, off_v8, off_v8};
          float a1b[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const uint32_t x = vwa[w];
            mma_bf16(a1, qb[2 * w], nib_bf16_off(x), nib_bf16_off(x >> 4));
            mma_bf16(a1b, qb[2 * w + 1], nib_bf16_off(x >> 8),
                     nib_bf16_off(x >> 12));
          }
          const __half2 sv = u32_as_h2(sc.x);
          const float sv0 = __low2float(sv) * kLog2eRsqrtD;
          const float sv1 = __high2float(sv) * kLog2eRsqrtD;
          const float P0 = (a1[0] + a1b[0]) * sv0, P1 = (a1[1] + a1b[1]) * sv1;
          const float P2 = (a1[2] + a1b[2]) * sv0, P3 = (a1[3] + a1b[3]) * sv1;
          const __half2 h01 = __floats2half2_rn(P0, P1);
          const __half2 h23 = __floats2half2_rn(P2, P3);
          const uint32_t A2h[4] = {h2_as_u32(h01), h2_as_u32(h23), 0u, 0u};
          const uint32_t A2l[4] = {split_lo(h2_as_u32(h01), P0, P1),
                                   split_lo(h2_as_u32(h23), P2, P3), 0u, 0u};
          // K 0..7 carry the high halves, K 8..15 the low halves
          const uint32_t A2[4] = {A2h[0], A2h[1], A2l[0], A2l[1]};
          uint32_t bt0, bt1;
          i8x4_to_h2(cw, bt0, bt1);
          float l0[4], l1[4];
          mma_f16_z(l0, A2, bt0, bt0);
          mma_f16_z(l1, A2, bt1, bt1);
          const __half2 sc0 = u32_as_h2(sc.y), sc1 = u32_as_h2(sc.z);
          const float c0 = __low2float(sc0), c1 = __high2float(sc0);
          const float c8 = __low2float(sc1), c9 = __high2float(sc1);
          const float e = lse2_quad_fast(l0[0] * c0, l0[1] * c1, l1[0] * c8,
                                         l1[1] * c9);
          const float e8 = lse2_quad_fast(l0[2] * c0, l0[3] * c1, l1[2] * c8,
                                          l1[3] * c9);
          if ((p >> 1) == t4) {
            if (p & 1) {
              o1 = e;
              o81 = e8;
            } else {
              o0 = e;
              o80 = e8;
            }
          }
        }
      }
      // q . mu for the tile's 8 pages (column n = page gq of the tile)
      float qm[4] = {off_m, off_m, off_m8, off_m8};
      float qm2[4] = {0.f, 0.f, 0.f, 0.f};
      {
        const uint32_t mrow = base_s + gq * kRec + kOffMu8 + 32 * t4;
        const uint4 m0 = lds128(mrow), m1 = lds128(mrow + 16);
        const uint32_t mw[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          uint32_t b01, b23;
          i8x4_to_h2_off(mw[s], b01, b23);
          if (s & 1)
            mma_f16(qm2, qh[s], b01, b23);
          else
            mma_f16(qm, qh[s], b01, b23);
        }
      }
      const int pg0 = 2 * t4, pg1 = 2 * t4 + 1;
      const float sm0 = __half2float(__ushort_as_half(
          (unsigned short)lds16(base_s + pg0 * kRec + kOffSMu)));
      const float sm1 = __half2float(__ushort_as_half(
          (unsigned short)lds16(base_s + pg1 * kRec + kOffSMu)));
      if (gq < G) {
        float *dst = lane_row + page0;
        if (pg0 < npg)
          dst[pg0] = (o0 + (qm[0] + qm2[0]) * sm0 * mscale) * kLn2;
        if (pg1 < npg)
          dst[pg1] = (o1 + (qm[1] + qm2[1]) * sm1 * mscale) * kLn2;
      }
      if (gq + 8 < G) {
        float *dst = lane_row8 + page0;
        if (pg0 < npg)
          dst[pg0] = (o80 + (qm[2] + qm2[2]) * sm0 * mscale) * kLn2;
        if (pg1 < npg)
          dst[pg1] = (o81 + (qm[3] + qm2[3]) * sm1 * mscale) * kLn2;
      }
    }
    __syncwarp();
    if (it + 2 < n_tiles) {
      issue_tile(nxt, nfull, summaries, h_kv, max_pages,
                 my_ring + stage * kTileBytes, &my_bar[stage], lane);
      advance_cursor(nxt, tph, batch, h_kv);
    }
    advance_cursor(cur, tph, batch, h_kv);
  }
  if (failed) {
    if (lane == 0) set_status(status, LOCKS_DEV_TIMEOUT);
    // let copies still in flight land before the CTA's memory goes away
    mbar_wait(&my_bar[0], 0, 1u << 16);
    mbar_wait(&my_bar[1], 0, 1u << 16);
    mbar_wait(&my_bar[0], 1, 1u << 16);
    mbar_wait(&my_bar[1], 1, 1u << 16);
  }
  if constexpr (FUSED)
    fused_select_epilogue<MODE>(nr, ns, s_hat, seq_lens, h_kv, G, max_pages,
                                k, fu_b, fu_h, fu_rank, fu_size,
                                tph[fu_b], smem, idx_out, status);
}

// --------------------------------------------------------------------------
// launchers
// --------------------------------------------------------------------------
size_t score_smem_bytes(int batch) {
  return (size_t)kRingBytes + sizeof(uint64_t) * kScoreWarps * kStages +
         sizeof(int) * (3 * (size_t)batch + 1);
}

int score_max_batch() {
  // the per-sequence tables must fit next to the ring in 227 KB
  return (int)((227 * 1024 - (size_t)kRingBytes -
                sizeof(uint64_t) * kScoreWarps * kStages - 64) /
               (3 * sizeof(int)));
}

cudaError_t launch_score(const void *q, const void *summaries,
                         const int32_t *seq_lens, int batch, int h_kv, int G,
                         int max_pages, float *s_hat, int32_t *status,
                         cudaStream_t stream, bool after_query) {
  const size_t smem = score_smem_bytes(batch);
  static DeviceFlags attr_set;
  cudaError_t ea = once_per_device(attr_set, [] {
    cudaError_t e = cudaFuncSetAttribute(
        score_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
        227 * 1024);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(score_kernel<2>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               227 * 1024);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(score_kernel<3>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               227 * 1024);
    return e;
  });
  if (ea != cudaSuccess) return ea;
  const int grid = device_sm_count();
  auto *qq = static_cast<const __nv_bfloat16 *>(q);
  auto *ss = static_cast<const uint8_t *>(summaries);
  auto *kern = G > 8 ? score_kernel<3> : G > 4 ? score_kernel<2>
                                               : score_kernel<1>;
  if (after_query)
    return launch_pdl(kern, dim3(grid), dim3(kScoreThreads), smem, stream, qq,
                      ss, seq_lens, batch, h_kv, G, max_pages, s_hat, status,
                      1, 0, (int32_t *)nullptr);
  kern<<<grid, kScoreThreads, smem, stream>>>(qq, ss, seq_lens, batch, h_kv, G,
                                              max_pages, s_hat, status, 0, 0,
                                              nullptr);
  return launched();
}

static_assert(kScoreThreads == kSelThreads,
              "the fused form runs select_top on the scoring block");

static cudaError_t fused_attributes() {
  static DeviceFlags attr_set;
  return once_per_device(attr_set, [] {
    cudaError_t e = cudaFuncSetAttribute(
        score_kernel<1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
        227 * 1024);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(score_kernel<2, true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               227 * 1024);
    return e;
  });
}

int fused_cluster_size(int batch, int h_kv, int G, int max_pages) {
  if (G > 8 || max_pages > kFusedMaxPages || batch > score_max_batch())
    return 0;
  if (fused_attributes() != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  const long long units = (long long)batch * h_kv;
  const int sms = device_sm_count();
  if (units < 1 || units > sms) return 0;
  int C = 8;
  while (C > 1 && units * C > sms) C >>= 1;
  // every cluster must be resident at once (one CTA per SM, C SMs of a
  // GPC each): ask the occupancy calculator, once per device and form
  static DeviceFlags fits[2][4];
  const int form = G > 4 ? 1 : 0;
  int lc = 0;
  for (int c = C; c > 1; c >>= 1) ++lc;
  for (; C >= 1; C >>= 1, --lc) {
    const int maxc = per_device_value(fits[form][lc], [&] {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)(units * C));
      cfg.blockDim = dim3(kScoreThreads);
      cfg.dynamicSmemBytes = score_smem_bytes(batch);
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = C;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(
              &n, form ? score_kernel<2, true> : score_kernel<1, true>,
              &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
      }
      return n + 1;  // cached values are >= 1
    });
    if (maxc - 1 >= units) return C;
  }
  return 0;
}

cudaError_t launch_score_select_fused(const void *q, const void *summaries,
                                      const int32_t *seq_lens, int batch,
                                      int h_kv, int G, int max_pages, int k,
                                      int cluster, float *s_hat, int32_t *idx,
                                      int32_t *status, cudaStream_t stream,
                                      bool after_query) {
  const cudaError_t ea = fused_attributes();
  if (ea != cudaSuccess) return ea;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((long long)batch * h_kv * cluster));
  cfg.blockDim = dim3(kScoreThreads);
  cfg.dynamicSmemBytes = score_smem_bytes(batch);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = after_query ? 2 : 1;
  auto *qq = static_cast<const __nv_bfloat16 *>(q);
  auto *ss = static_cast<const uint8_t *>(summaries);
  const cudaError_t e = cudaLaunchKernelEx(
      &cfg, G > 4 ? score_kernel<2, true> : score_kernel<1, true>, qq, ss,
      seq_lens, batch, h_kv, G, max_pages, s_hat, status,
      after_query ? 1 : 0, k, idx);
  if (e == cudaSuccess) note_launches();
  return e;
}

}  // namespace locks
