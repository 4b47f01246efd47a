// Attention over the selected pages (LOCKS reading notes §2 and §4.4
// Algorithm 2: fetch full K/V only for the selected pages, then standard
// softmax attention for every query head of the group).
//
// Warp-streamed flash decode.  The page lists of all (sequence, KV head)
// units are laid end to end (a "position" is one entry of one unit's list:
// idx[b][h][i] for sparse decode, page i of sequence b for dense decode) and
// every warp of a grid sized to fill the GPU takes one contiguous run of
// `chunk` positions, so all warps stream the same number of pages whatever
// the list lengths.  A warp resolves 32 positions at a time (index -> page
// table -> physical page, one per lane), gathers each valid page (one 4 KB
// K run and one 4 KB V run) with 16-byte cp.async into a private,
// double-buffered, XOR-swizzled shared-memory tile, and runs Q K^T and P V on
// bf16 mma.sync with the query heads as the M dimension; every K/V byte is
// read once for the whole GQA group.  Softmax is online in base 2.
//
// A unit that lies inside one warp's run is finished by that warp.  A unit
// split across warps leaves one normalised partial (o, lse) per warp in
// slot (unit + warp) -- distinct for distinct (unit, warp) pieces because
// both grow along the positions -- and a second small kernel merges them.
//
// Unit form (sparse decode): every unit has exactly k list positions, so a
// cluster of C CTAs takes one unit (C = 1 with at least one unit per SM),
// its 4C warps a slice of the list each with a three-stage ring (two CTAs
// per SM: the same 24 pages in flight per SM), and the 4C partials are
// merged at the end in shared memory, across the cluster through
// distributed shared memory: no partials in the workspace and no merge
// launch.
#include "common.cuh"
#include "launch.h"

namespace locks {

constexpr int kDecWarps = 4;
constexpr int kDecThreads = 32 * kDecWarps;
constexpr int kDecStages = 2;
constexpr int kKvTile = kPage * kDim * 2;                          // 4096 B
constexpr int kDecRing = kDecWarps * kDecStages * 2 * kKvTile;      // 64 KB
// resident CTAs per SM the register budget is sized for (G > 8 keeps a
// second row of accumulators and takes two)
constexpr int kDecMinBlocks = 3;
// Sparse decode: fewest list positions per warp.  Graph-replayed decode +
// merge on GB300: 64 units x 128 pages (G = 8) 17.5 -> 14.0 us, 64 x 64
// (G = 4) 11.6 -> 10.5 us; 256 x 128 unchanged (already above 8 per warp).
constexpr int kDecMinRun = 8;
constexpr int kDecUnitStages = 3;  // unit form: stages per warp
constexpr int kDecClusterMinRun = 1;  // unit form in clusters: positions per warp
constexpr float kDecScale = 0.12751743074602467f;  // log2(e)/sqrt(d)
constexpr float kLn2f = 0.69314718055994531f;

__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

// swizzled byte offset of 16-byte chunk `ch` (0..15) of token row `row`
__device__ __forceinline__ uint32_t swz(int row, int ch) {
  return (uint32_t)(row * 256 + ((ch ^ (row & 7)) << 4));
}

// Position layout shared by the two kernels.  Sequence b's h_kv units are
// consecutive, each len_b positions long, and start at position first(b):
// b * h_kv * k for sparse decode (per_seq = h_kv * k), pre[b] (a prefix sum
// over the sequences' page counts) for dense decode (per_seq = 0).
struct Layout {
  const int *pre;
  int batch, h_kv, per_seq;

  __device__ __forceinline__ int first(int b) const {
    return per_seq ? b * per_seq : pre[b];
  }
  // sequence holding position p (p below the total)
  __device__ __forceinline__ int seq(int p) const {
    if (per_seq) return p / per_seq;
    int lo = 0, hi = batch;  // largest b with pre[b] <= p
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (pre[mid] <= p) lo = mid; else hi = mid;
    }
    return lo;
  }
  __device__ __forceinline__ int unit_len(int b) const {
    return (first(b + 1) - first(b)) / h_kv;
  }
  __device__ __forceinline__ int unit_of(int p) const {
    const int b = seq(p);
    return b * h_kv + (p - first(b)) / unit_len(b);
  }
  // positions [begin, end) of unit u
  __device__ __forceinline__ int2 span(int u) const {
    const int b = u / h_kv, h = u - b * h_kv;
    const int f = first(b), len = unit_len(b);
    return make_int2(f + h * len, f + (h + 1) * len);
  }
};

__device__ __forceinline__ int clamp_len(const int32_t *seq_lens, int b,
                                         int max_pages, int32_t *status) {
  int L = __ldg(seq_lens + b);
  if (L < 0 || L > max_pages * kPage) {
    set_status(status, LOCKS_DEV_BAD_SEQ_LEN);
    L = max(0, min(L, max_pages * kPage));
  }
  return L;
}

// One lane's entry of a 32-position window.
struct Entry {
  int phys;  // physical page, -1 when the position is skipped
  int ntok;  // tokens of the page inside the sequence
  int u;     // unit (b * h_kv + h)
};

__device__ __forceinline__ Entry resolve(int p, int pe, const Layout &lay,
                                         const int32_t *seq_lens,
                                         const int32_t *idx, int k,
                                         const int32_t *pt, int max_pages,
                                         int64_t num_phys, int32_t *status) {
  Entry e{-1, 0, 0};
  if (p >= pe) return e;
  const int b = lay.seq(p);
  const int len = lay.unit_len(b);
  const int r = p - lay.first(b);
  const int h = r / len, slot = r - h * len;
  e.u = b * lay.h_kv + h;
  const int L = clamp_len(seq_lens, b, max_pages, status);
  const int n = (L + kPage - 1) / kPage;
  const int pg = idx ? __ldg(idx + (size_t)e.u * k + slot) : slot;
  if (pg >= n) {
    set_status(status, LOCKS_DEV_BAD_INDEX);
  } else if (pg >= 0) {
    const int ph = __ldg(pt + (size_t)b * max_pages + pg);
    if (ph < 0 || ph >= num_phys) {
      set_status(status, LOCKS_DEV_BAD_PAGE_ID);
    } else {
      e.phys = ph;
      e.ntok = min(kPage, L - pg * kPage);
    }
  }
  return e;
}

template <bool WIDE, bool UNIT = false>
__global__ void __launch_bounds__(kDecThreads,
                                  UNIT ? 2 : (WIDE ? 2 : kDecMinBlocks))
    decode_kernel(const __nv_bfloat16 *__restrict__ q,
                  const __nv_bfloat16 *__restrict__ k_cache,
                  const __nv_bfloat16 *__restrict__ v_cache, int64_t num_phys,
                  const int32_t *__restrict__ pt,
                  const int32_t *__restrict__ seq_lens,
                  const int32_t *__restrict__ idx, int k, int batch, int h_kv,
                  int G, int max_pages, int n_warps,
                  __nv_bfloat16 *__restrict__ o_out,
                  float *__restrict__ lse_out, float *__restrict__ o_part,
                  float *__restrict__ lse_part, int *__restrict__ meta,
                  int32_t *status) {
  constexpr int STG = UNIT ? kDecUnitStages : kDecStages;
  constexpr int kWarpRing = STG * 2 * kKvTile;
  extern __shared__ __align__(128) uint8_t smem[];
  int *s_pre =
      reinterpret_cast<int *>(smem + kDecWarps * kWarpRing);  // [batch + 1]
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int gq = lane >> 2, t4 = lane & 3;
  const int h_q = h_kv * G;
  const Layout lay{s_pre, batch, h_kv, idx ? h_kv * k : 0};
  pdl_trigger();

  int total;
  if (idx) {
    total = batch * h_kv * k;
  } else {
    // dense: h_kv lists of the sequence's page count; inclusive scan into
    // s_pre[1..batch]
    for (int b = threadIdx.x; b < batch; b += blockDim.x) {
      const int L = clamp_len(seq_lens, b, max_pages,
                              blockIdx.x == 0 ? status : nullptr);
      s_pre[b + 1] = h_kv * ((L + kPage - 1) / kPage);
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
    total = s_pre[batch];
  }
  const int chunk =
      (int)max(1LL, ((long long)total + n_warps - 1) / n_warps);
  const int gw = blockIdx.x * kDecWarps + wid;
  bool active;
  int pb, pe;
  // unit form: CTAs per unit (the cluster) and this CTA's rank in it
  const int ucl = UNIT ? (int)cluster_nctarank() : 1;
  const int urank = UNIT && ucl > 1 ? (int)cluster_ctarank() : 0;
  if constexpr (UNIT) {  // slice urank * 4 + wid of the unit's k positions
    const int u0 = (int)blockIdx.x / ucl;
    const int sl = urank * kDecWarps + wid, nsl = ucl * kDecWarps;
    pb = u0 * k + (int)((long long)sl * k / nsl);
    pe = u0 * k + (int)((long long)(sl + 1) * k / nsl);
    active = pe > pb;
  } else {
    active = gw < n_warps && (long long)gw * chunk < total;
    pb = active ? gw * chunk : 0;
    pe = min(total, pb + chunk);
  }

  uint8_t *wbase = smem + wid * kWarpRing;
  const uint32_t wbase_s = smem_u32(wbase);

  // query A fragments (bf16) of unit u, rows = heads of the group
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
  // the query is an input of the step: fetch it while the selection kernel
  // may still run
  int cur_u = UNIT ? (int)blockIdx.x / ucl : active ? lay.unit_of(pb) : 0;
  if (active) load_q(cur_u);
  // the page lists come from the selection kernel, and the workspace may
  // still be read by it
  pdl_wait();
  if (!UNIT && blockIdx.x == 0) {  // layout for the merge kernel
    if (threadIdx.x == 0) meta[0] = chunk;
    if (!idx)
      for (int b = threadIdx.x; b <= batch; b += blockDim.x)
        meta[1 + b] = s_pre[b];
  }
  // (unit form: an empty quarter still takes part in the CTA's merge)
  if (!UNIT && !active) return;
  bool q_ready = true;

  // window of 32 positions: this lane's entry and the valid ones not yet
  // handed to the copy engine
  int win = pb - 32;
  uint32_t wmask = 0;
  Entry we{-1, 0, 0};
  // next valid position in order (phys < 0: none left)
  auto next_valid = [&](int &phys, int &ntok, int &u) {
    while (wmask == 0) {
      win += 32;
      if (win >= pe) {
        phys = -1;
        return;
      }
      we = resolve(win + lane, pe, lay, seq_lens, idx, k, pt, max_pages,
                   num_phys, status);
      wmask = __ballot_sync(0xffffffffu, we.phys >= 0);
    }
    const int j = __ffs(wmask) - 1;
    wmask &= wmask - 1;
    phys = __shfl_sync(0xffffffffu, we.phys, j);
    ntok = __shfl_sync(0xffffffffu, we.ntok, j);
    u = __shfl_sync(0xffffffffu, we.u, j);
  };
  auto issue = [&](int stage, int phys, int u) {
    const int h = u % h_kv;
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

  // write unit u's result (whole unit inside this run) or partial (slot
  // u + gw), then reset the accumulators
  auto flush = [&](int u) {
    float l = l_run, l8 = l_run8;
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    l8 += __shfl_xor_sync(0xffffffffu, l8, 1);
    l8 += __shfl_xor_sync(0xffffffffu, l8, 2);
    const int2 sp = lay.span(u);
    const bool whole = !UNIT && sp.x >= pb && sp.y <= pe;
    const int b = u / h_kv, h = u - b * h_kv;
#pragma unroll
    for (int half = 0; half < (WIDE ? 2 : 1); ++half) {
      const int g = gq + 8 * half;
      const float lh = half ? l8 : l;
      const float mh = half ? m_run8 : m_run;
      const float inv = lh > 0.f ? 1.f / lh : 0.f;
      const float lse = lh > 0.f ? (mh + log2f(lh)) * kLn2f : -INFINITY;
      if (g < G) {
        if (whole) {
          const size_t row = (size_t)b * h_q + (size_t)h * G + g;
          uint32_t *dst = reinterpret_cast<uint32_t *>(o_out + row * kDim);
#pragma unroll
          for (int nt = 0; nt < 16; ++nt)
            dst[(nt * 8 + 2 * t4) >> 1] =
                pack_bf2(o[nt][2 * half] * inv, o[nt][2 * half + 1] * inv);
          if (t4 == 0) lse_out[row] = lse;
        } else {
          // partial: slot (unit + warp) of the workspace, or (unit form)
          // row g of this warp's ring region, drained by then
          float *po = UNIT ? reinterpret_cast<float *>(wbase) + g * kDim
                           : o_part + (((size_t)u + gw) * G + g) * kDim;
          float *pl = UNIT ? reinterpret_cast<float *>(wbase) + 16 * kDim + g
                           : lse_part + ((size_t)u + gw) * G + g;
          float2 *dst = reinterpret_cast<float2 *>(po);
#pragma unroll
          for (int nt = 0; nt < 16; ++nt)
            dst[(nt * 8 + 2 * t4) >> 1] =
                make_float2(o[nt][2 * half] * inv, o[nt][2 * half + 1] * inv);
          if (t4 == 0) *pl = lse;
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    m_run = m_run8 = -INFINITY;
    l_run = l_run8 = 0.f;
  };
  // close every unit before `u` (units with no positions are the merge
  // kernel's)
  auto advance_to = [&](int u) {
    while (cur_u < u) {
      const int2 sp = lay.span(cur_u);
      if (sp.y > sp.x) flush(cur_u);
      ++cur_u;
      q_ready = false;
    }
  };

  // pages in flight, oldest first (qp < 0: none); the oldest sits in shared
  // memory stage `st`, the next ones in the stages after it
  int qp[STG], qn[STG], qu[STG];
#pragma unroll
  for (int i = 0; i < STG; ++i) {
    qn[i] = 0;
    qu[i] = 0;
    next_valid(qp[i], qn[i], qu[i]);
    if (qp[i] >= 0) issue(i, qp[i], qu[i]);
    cp_async_commit();
  }

  for (int st = 0;; st = st + 1 == STG ? 0 : st + 1) {
    const int phys = qp[0];
    if (phys < 0) break;
    const int ntok = qn[0];
    const int u = qu[0];
    if (u != cur_u) advance_to(u);
    if (!q_ready) {
      load_q(cur_u);
      q_ready = true;
    }
    cp_async_wait<STG - 1>();
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
#pragma unroll
    for (int i = 0; i + 1 < STG; ++i) {
      qp[i] = qp[i + 1];
      qn[i] = qn[i + 1];
      qu[i] = qu[i + 1];
    }
    qn[STG - 1] = 0;
    qu[STG - 1] = 0;
    next_valid(qp[STG - 1], qn[STG - 1], qu[STG - 1]);
    if (qp[STG - 1] >= 0) issue(st, qp[STG - 1], qu[STG - 1]);
    cp_async_commit();
  }
  cp_async_wait<0>();
  __syncwarp();
  if constexpr (!UNIT) {
    // close the units up to the one holding the run's last position
    const int u_last = lay.unit_of(pe - 1);
    advance_to(u_last);
    flush(u_last);
  } else {
    // the 4C slices of the unit, merged row by row: CTA r of the cluster
    // takes heads r, r + C, ..., warp w of it every fourth of those; lane l
    // dims 4l .. 4l + 3.  Slice (c, w) is warp w's ring region in CTA c.
    const int u = (int)blockIdx.x / ucl;
    flush(u);
    if (ucl > 1)
      cluster_sync();
    else
      __syncthreads();
    const int b = u / h_kv, h = u - b * h_kv;
    const int nsl = ucl * kDecWarps;
    const uint32_t base_s = smem_u32(smem);
    // shared::cluster address of float `i` of slice s's region
    auto at = [&](int s2, int i) -> uint32_t {
      return mapa_shared(
          base_s + (uint32_t)((s2 % kDecWarps) * kWarpRing + 4 * i),
          (uint32_t)(s2 / kDecWarps));
    };
    constexpr int kMaxSlices = 8 * kDecWarps;  // clusters of up to 8 CTAs
    for (int g = urank + ucl * wid; g < G; g += ucl * kDecWarps) {
      const size_t row = (size_t)b * h_q + (size_t)h * G + g;
      uint2 *dst = reinterpret_cast<uint2 *>(o_out + row * kDim) + lane;
      float wsum = 0.f, M = -INFINITY;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      if (ucl == 1) {  // the CTA's own four slices
        float l[kDecWarps];
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) {
          l[w] = reinterpret_cast<const float *>(smem + w * kWarpRing)[16 * kDim + g];
          M = fmaxf(M, l[w]);
        }
        if (M > -INFINITY) {
#pragma unroll
          for (int w = 0; w < kDecWarps; ++w) {
            if (l[w] == -INFINITY) continue;
            const float f = expf(l[w] - M);
            const float4 v = reinterpret_cast<const float4 *>(
                smem + w * kWarpRing)[g * (kDim / 4) + lane];
            wsum += f;
            acc.x += f * v.x;
            acc.y += f * v.y;
            acc.z += f * v.z;
            acc.w += f * v.w;
          }
        }
      } else {  // every slice of the cluster: all loads issued before use
        float l[kMaxSlices];
#pragma unroll
        for (int s2 = 0; s2 < kMaxSlices; ++s2)
          l[s2] = s2 < nsl ? ld_cluster_f32(at(s2, 16 * kDim + g)) : -INFINITY;
#pragma unroll
        for (int s2 = 0; s2 < kMaxSlices; ++s2) M = fmaxf(M, l[s2]);
        if (M > -INFINITY) {
#pragma unroll
          for (int h0 = 0; h0 < kMaxSlices; h0 += 16) {
            float4 v[16];
#pragma unroll
            for (int j = 0; j < 16; ++j)
              v[j] = h0 + j < nsl && l[h0 + j] > -INFINITY
                         ? ld_cluster_v4f(at(h0 + j, g * kDim + 4 * lane))
                         : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float f =
                  l[h0 + j] > -INFINITY ? expf(l[h0 + j] - M) : 0.f;
              wsum += f;
              acc.x += f * v[j].x;
              acc.y += f * v[j].y;
              acc.z += f * v[j].z;
              acc.w += f * v[j].w;
            }
          }
        }
      }
      if (M == -INFINITY) {  // no tokens
        *dst = make_uint2(0u, 0u);
        if (lane == 0) lse_out[row] = -INFINITY;
        continue;
      }
      const float inv = 1.f / wsum;
      *dst = make_uint2(pack_bf2(acc.x * inv, acc.y * inv),
                        pack_bf2(acc.z * inv, acc.w * inv));
      if (lane == 0) lse_out[row] = M + logf(wsum);
    }
    // no CTA leaves while another may still read its slices
    if (ucl > 1) cluster_sync();
  }
}

// the step's device status word, copied where the host reads it once the
// decode kernel is done (unit form, which launches no merge kernel)
__global__ void status_mirror_kernel(const int32_t *__restrict__ src,
                                     int32_t *dst) {
  pdl_wait();
  *dst = *src;
}

// Merge of the partials of units split across warps; also writes the
// empty result of units with no positions.  One warp per (unit, head) row;
// lane l owns head dimensions 4l..4l+3.  Pieces are merged eight at a time
// with an online rescale, all loads of a group issued together, so a unit
// split across at most eight warps costs one round trip.
constexpr int kCombineWarps = 4;
constexpr int kCombineGroup = 8;

__global__ void __launch_bounds__(32 * kCombineWarps)
    combine_kernel(const float *__restrict__ o_part,
                   const float *__restrict__ lse_part,
                   const int *__restrict__ meta, int batch, int h_kv, int k,
                   int dense, int G, __nv_bfloat16 *__restrict__ o_out,
                   float *__restrict__ lse_out,
                   const int32_t *__restrict__ status_src,
                   int32_t *status_mirror, int chunk_hint) {
  const int lane = threadIdx.x & 31;
  pdl_wait();  // partials and layout of the decode kernel
  // the step's device status word is final once the decode kernel is done
  // (every kernel before it waited on its predecessor): copy it out
  if (status_mirror && blockIdx.x == 0 && threadIdx.x == 0)
    *status_mirror = *status_src;
  const long long row =
      (long long)blockIdx.x * kCombineWarps + (threadIdx.x >> 5);
  if (row >= (long long)batch * h_kv * G) return;
  const int u = (int)(row / G), g = (int)(row - (long long)u * G);
  const Layout lay{meta + 1, batch, h_kv, dense ? 0 : h_kv * k};
  // sparse decode: the run length is known at launch (saves a dependent
  // load); dense decode reads it from the decode kernel's layout
  const int chunk = chunk_hint > 0 ? chunk_hint : meta[0];
  const int2 sp = lay.span(u);
  uint2 *dst = reinterpret_cast<uint2 *>(o_out + row * kDim) + lane;
  float M = -INFINITY, wsum = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (sp.y > sp.x) {
    const int w0 = sp.x / chunk, w1 = (sp.y - 1) / chunk;
    if (w0 == w1) return;  // finished by its warp
    const float4 *o4 = reinterpret_cast<const float4 *>(o_part);
    for (int wb = w0; wb <= w1; wb += kCombineGroup) {
      float l[kCombineGroup];
      float4 v[kCombineGroup];
#pragma unroll
      for (int j = 0; j < kCombineGroup; ++j) {
        const size_t slot = ((size_t)u + wb + j) * G + g;
        const bool in = wb + j <= w1;
        l[j] = in ? lse_part[slot] : -INFINITY;
        v[j] = in ? o4[slot * 32 + lane] : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      float gm = l[0];
#pragma unroll
      for (int j = 1; j < kCombineGroup; ++j) gm = fmaxf(gm, l[j]);
      const float Mn = fmaxf(M, gm);
      if (Mn == -INFINITY) continue;
      const float cf = M == -INFINITY ? 0.f : expf(M - Mn);
      wsum *= cf;
      acc.x *= cf;
      acc.y *= cf;
      acc.z *= cf;
      acc.w *= cf;
#pragma unroll
      for (int j = 0; j < kCombineGroup; ++j) {
        const float f = l[j] == -INFINITY ? 0.f : expf(l[j] - Mn);
        wsum += f;
        acc.x += f * v[j].x;
        acc.y += f * v[j].y;
        acc.z += f * v[j].z;
        acc.w += f * v[j].w;
      }
      M = Mn;
    }
  }
  if (M == -INFINITY) {  // no tokens
    *dst = make_uint2(0u, 0u);
    if (lane == 0) lse_out[row] = -INFINITY;
    return;
  }
  const float inv = 1.f / wsum;
  *dst = make_uint2(pack_bf2(acc.x * inv, acc.y * inv),
                    pack_bf2(acc.z * inv, acc.w * inv));
  if (lane == 0) lse_out[row] = M + logf(wsum);
}

// --------------------------------------------------------------------------
// launchers
// --------------------------------------------------------------------------
size_t decode_smem_bytes(int batch) {
  return (size_t)kDecRing + sizeof(int) * ((size_t)batch + 1);
}

// the unit form keeps only the warps' rings (no per-sequence table: it is
// sparse decode only), so its footprint does not grow with the batch
static size_t decode_unit_smem_bytes() {
  return (size_t)kDecWarps * kDecUnitStages * 2 * kKvTile;
}

int decode_max_batch() {
  return (int)((227 * 1024 - (size_t)kDecRing - 64) / sizeof(int));
}

cudaError_t launch_decode(const void *q, const void *k_cache,
                          const void *v_cache, int64_t num_phys,
                          const int32_t *pt, const int32_t *seq_lens,
                          const int32_t *idx, int k, int batch, int h_kv,
                          int G, int max_pages, int max_warps, void *o_out,
                          float *lse_out, float *o_part, float *lse_part,
                          int *meta, int32_t *status, cudaStream_t stream,
                          int32_t *status_mirror) {
  static DeviceFlags attr_set, blocks_narrow, blocks_wide;
  cudaError_t ea = once_per_device(attr_set, [] {
    cudaError_t e = cudaFuncSetAttribute(
        decode_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
        227 * 1024);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(decode_kernel<true>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                227 * 1024);
  });
  if (ea != cudaSuccess) return ea;
  const size_t smem = decode_smem_bytes(batch);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  const int wide = G > 8 ? 1 : 0;
  auto *qq = static_cast<const __nv_bfloat16 *>(q);
  auto *kc = static_cast<const __nv_bfloat16 *>(k_cache);
  auto *vc = static_cast<const __nv_bfloat16 *>(v_cache);
  auto *oo = static_cast<__nv_bfloat16 *>(o_out);
  // unit form: sparse decode with every SM holding at least one unit, or a
  // cluster of 8 or 4 CTAs per unit when all of them fit two per SM and
  // every warp has a list position.  Graph-replayed decode on GB300 against
  // the split form and its merge: 64 units x 128 pages (G = 8, clusters of
  // 4) 14.1 -> 12.7 us, 64 x 64 (G = 4, clusters of 4) 10.5 -> 9.1 us,
  // 2 x 16 (clusters of 4, one page per warp) 6.7 -> 6.3 us and the whole
  // step 19.7 -> 17.5 us (no merge launch on the chain); clusters of 2 lost
  // (11.2 against 10.5 us).
  const long long units = (long long)batch * h_kv;
  const int sms = device_sm_count();
  int ucl = 0;
  if (idx && units <= 0x7fffffffLL / (8 * kDecWarps)) {
    if (units >= sms) {
      ucl = 1;
    } else {
      for (int c = 8; c >= 4 && !ucl; c >>= 1)
        if (units * c <= 2LL * sms && k >= c * kDecWarps * kDecClusterMinRun)
          ucl = c;
    }
  }
  if (ucl > 0) {
    static DeviceFlags unit_attr;
    cudaError_t eu = once_per_device(unit_attr, [] {
      cudaError_t e = cudaFuncSetAttribute(
          decode_kernel<false, true>,
          cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
      if (e != cudaSuccess) return e;
      return cudaFuncSetAttribute(decode_kernel<true, true>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  227 * 1024);
    });
    if (eu != cudaSuccess) return eu;
    const size_t usmem = decode_unit_smem_bytes();
    auto *ukern = wide ? decode_kernel<true, true> : decode_kernel<false, true>;
    const dim3 ugrid((unsigned)(units * ucl));
    const int uwarps = (int)(units * ucl * kDecWarps);
    cudaError_t e =
        ucl > 1 ? launch_pdl_cluster(ukern, ugrid, dim3(kDecThreads), usmem,
                                     stream, ucl, qq, kc, vc, num_phys, pt,
                                     seq_lens, idx, k, batch, h_kv, G,
                                     max_pages, uwarps, oo, lse_out, o_part,
                                     lse_part, meta, status)
                : launch_pdl(ukern, ugrid, dim3(kDecThreads), usmem, stream,
                             qq, kc, vc, num_phys, pt, seq_lens, idx, k,
                             batch, h_kv, G, max_pages, uwarps, oo, lse_out,
                             o_part, lse_part, meta, status);
    if (e != cudaSuccess || !status_mirror) return e;
    return launch_pdl(status_mirror_kernel, dim3(1), dim3(1), 0, stream,
                      (const int32_t *)status, status_mirror);
  }
  // resident CTAs per SM at the common (small-batch) footprint; a larger
  // batch only lowers the count the hardware actually fits
  const int blocks_per_sm =
      per_device_value(wide ? blocks_wide : blocks_narrow, [wide] {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                &n, wide ? decode_kernel<true> : decode_kernel<false>,
                kDecThreads, decode_smem_bytes(64)) != cudaSuccess)
          return 0;
        return n;
      });
  long long warps = (long long)blocks_per_sm * device_sm_count() * kDecWarps;
  if (warps > max_warps) warps = max_warps;
  if (idx) {
    // at least kDecMinRun list positions per warp, so that a unit is split
    // into fewer pieces for the merge, unless that leaves fewer than two
    // warps per SM
    long long cap = ((long long)batch * h_kv * k + kDecMinRun - 1) / kDecMinRun;
    if (cap < 2LL * device_sm_count()) cap = 2LL * device_sm_count();
    if (warps > cap) warps = cap;
  }
  if (warps < 1) warps = 1;
  const int n_warps = (int)warps;
  const int grid = (n_warps + kDecWarps - 1) / kDecWarps;
  cudaError_t e = launch_pdl(
      wide ? decode_kernel<true> : decode_kernel<false>, dim3(grid),
      dim3(kDecThreads), smem, stream, qq, kc, vc, num_phys, pt, seq_lens,
      idx, k, batch, h_kv, G, max_pages, n_warps, oo, lse_out, o_part,
      lse_part, meta, status);
  if (e != cudaSuccess) return e;
  const long long rows = (long long)batch * h_kv * G;
  // the decode kernel's run length for sparse decode (dense decode's
  // depends on the sequence lengths and is read on the device)
  const long long per_warp =
      ((long long)batch * h_kv * k + n_warps - 1) / n_warps;
  const int chunk_hint = idx ? (int)(per_warp > 1 ? per_warp : 1) : 0;
  return launch_pdl(combine_kernel,
                    dim3((unsigned)((rows + kCombineWarps - 1) / kCombineWarps)),
                    dim3(32 * kCombineWarps), 0, stream, o_part, lse_part,
                    (const int *)meta, batch, h_kv, k, idx ? 0 : 1, G, oo,
                    lse_out, (const int32_t *)status, status_mirror,
                    chunk_hint);
}

}  // namespace locks
