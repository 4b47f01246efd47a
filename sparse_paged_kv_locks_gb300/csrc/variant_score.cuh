// Scoring from rank / precision variant records (LOCKS reading notes §4.2
// Eq.(4) with the §6 ablation's ranks and basis precisions):
//   s_hat_j(q_g) = ln sum_{i<16} exp((q_g . mu_j + (V_j^T q_g) . c_i) / sqrt(d))
// for records laid out as variant_layout.cuh describes.
//
// The same streaming design as the shipped scorer: a persistent grid, one
// contiguous range of tiles (TP records of one (sequence, KV head)) per
// warp, tiles double-buffered in shared memory by 1-D bulk copies on
// mbarriers, all arithmetic on mma.sync with fp16 operands:
//   product 1 (transposed)  D[row][n] = sum_d code[row][d] q_n[d] / scale
//       rows: the basis components of PG pages (PG = 16 / rows per page),
//       A fragments unpacked straight from the lane's slot words (the code
//       offset is cancelled through the accumulator's initial value)
//   product 2               L[g][i] = sum_k P[g][k] C[i][k], P = D sV split
//       into high and low fp16 halves, turned head-major with movmatrix
//   product 3               q_g . mu_p for the TP pages of the tile
// then the 16-token log-sum-exp per (page, head) over a lane quad.
// MODE 1 (G <= 4, PG >= 2) packs two pages into the rows of product 2;
// MODE 2 (G <= 8) keeps heads in rows 0..7 (high) and 8..15 (low);
// MODE 3 (G <= 16) runs product 2 of MODE 2 once per half of the heads.
#pragma once
#include "common.cuh"
#include "launch.h"
#include "score_ops.cuh"
#include "variant_layout.cuh"

namespace locks {

__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];\n"
               : "=r"(v.x), "=r"(v.y)
               : "r"(a));
  return v;
}

__device__ __forceinline__ float lds_f16(uint32_t a) {
  return __half2float(__ushort_as_half((unsigned short)lds16(a)));
}

// Product-1 A operand of k-step s, half h (h = 0: dims 16s + 0..7, h = 1:
// dims 16s + 8..15) from a lane's slot words, as fp16x2 holding
// offset(s, h) + scale(s, h) * code (exact); the query operand of those
// dims is divided by scale(s, h) and the offsets are cancelled through the
// accumulator's initial value.
template <int VB>
struct VCodes;

template <>
struct VCodes<4> {
  static constexpr int words = 4;
  __device__ static uint32_t op(const uint32_t (&w)[4], int s, int h) {
    const uint32_t x = (s & 1) ? w[s >> 1] >> 8 : w[s >> 1];
    return h ? nib_f16_hi(x) : nib_f16_lo(x);
  }
  __host__ __device__ static constexpr float scale(int, int h) {
    return h ? 16.f : 1.f;
  }
  __host__ __device__ static constexpr float offset(int, int h) {
    return h ? 1152.f : 1032.f;
  }
};

// 2-bit codes: position j = 2 (s % 4) + h of the half-word; positions 0..4
// sit at bits 2j (scale 4^j), 5..7 are shifted down by 10 first (scale
// 4^(j-5)); the code's sign bit is flipped, so the value is
// 1024 + scale * (code + 2).
template <>
struct VCodes<2> {
  static constexpr int words = 2;
  __host__ __device__ static constexpr int pos(int s, int h) {
    return 2 * (s & 3) + h < 5 ? 2 * (s & 3) + h : 2 * (s & 3) + h - 5;
  }
  __device__ static uint32_t op(const uint32_t (&w)[2], int s, int h) {
    const int j = 2 * (s & 3) + h, p = pos(s, h);
    const uint32_t x = j < 5 ? w[s >> 2] : w[s >> 2] >> 10;
    return lop3_and_xor(x, 0x00030003u << (2 * p),
                        0x64006400u | (0x00020002u << (2 * p)));
  }
  __host__ __device__ static constexpr float scale(int s, int h) {
    return (float)(1 << (2 * pos(s, h)));
  }
  __host__ __device__ static constexpr float offset(int s, int h) {
    return 1024.f + 2.f * scale(s, h);
  }
};

// 8-bit codes, excess-128: bytes (e, h) = (0,0), (1,0), (0,1), (1,1) of
// word s; 1024 + byte = 1152 + code
template <>
struct VCodes<8> {
  static constexpr int words = 8;
  __device__ static uint32_t op(const uint32_t (&w)[8], int s, int h) {
    uint32_t r;
    if (h)
      asm("prmt.b32 %0, %1, %2, 0x7372;\n" : "=r"(r) : "r"(w[s]), "r"(0x64646464u));
    else
      asm("prmt.b32 %0, %1, %2, 0x7170;\n" : "=r"(r) : "r"(w[s]), "r"(0x64646464u));
    return r;
  }
  __host__ __device__ static constexpr float scale(int, int) { return 1.f; }
  __host__ __device__ static constexpr float offset(int, int) {
    return 1152.f;
  }
};

template <int VB>
__device__ __forceinline__ void load_slot(uint32_t (&w)[VCodes<VB>::words],
                                          uint32_t a) {
  if constexpr (VB == 2) {
    const uint2 v = lds64(a);
    w[0] = v.x;
    w[1] = v.y;
  } else {
#pragma unroll
    for (int i = 0; i < VB / 4; ++i) {
      const uint4 v = lds128(a + 16 * i);
      w[4 * i] = v.x;
      w[4 * i + 1] = v.y;
      w[4 * i + 2] = v.z;
      w[4 * i + 3] = v.w;
    }
  }
}

// log-sum-exp (log2 units) of one page and head from product 2's two token
// tiles (rows gq: high halves, gq + 8: low halves) and the page's
// coefficient scales sC[2t4], sC[2t4+1], sC[8+2t4], sC[9+2t4]
__device__ __forceinline__ float var_page_lse(const float (&l0)[4],
                                              const float (&l1)[4],
                                              uint32_t sc_a, uint32_t sc_b,
                                              bool safe, uint32_t &bad) {
  const __half2 s0 = u32_as_h2(sc_a), s1 = u32_as_h2(sc_b);
  return lse2_quad_sel((l0[0] + l0[2]) * __low2float(s0),
                       (l0[1] + l0[3]) * __high2float(s0),
                       (l1[0] + l1[2]) * __low2float(s1),
                       (l1[1] + l1[3]) * __high2float(s1), safe, bad);
}

// The basis and coefficient products and the per-page log-sum-exp of one
// tile's pages, a product-1 group of PG pages per step.  keep[nt][u]:
// MODE 2/3: head gq + 8 nt, page 2 t4 + u; MODE 1: keep[0][0], head gq & 3,
// page 2 t4 + (gq >= 4).  SAFE selects the max-subtracted log-sum-exp;
// otherwise the return value folds every quad sum's distance from the
// normal range (>= kLseBad: recompute with SAFE).
template <int R, int VB, int MODE, bool SAFE>
__device__ __forceinline__ uint32_t var_score_groups(
    uint32_t base_s, int npg, int lane,
    const uint32_t (&qv)[MODE == 3 ? 2 : 1][8][2],
    const float (&offc)[MODE == 3 ? 2 : 1][2], float vscale,
    float (&keep)[MODE == 3 ? 2 : 1][2]) {
  using VC = VCodes<VB>;
  constexpr int NT = MODE == 3 ? 2 : 1;
  constexpr int ST = var_stride(R, VB), PG = var_pages_per_group(R);
  constexpr int OFF_C = var_off_c(R, VB), OFF_S = var_off_s(R, VB);
  static_assert(MODE != 1 || PG > 1, "MODE 1 pairs pages in product 2");
  const int gq = lane >> 2, t4 = lane & 3;
  // rows gq (X) and gq + 8 (Y) of the product-1 group: page and component
  const int xpage = PG == 4 ? gq >> 2 : 0;
  const int ypage = PG == 4 ? 2 + (gq >> 2) : PG == 2 ? 1 : 0;
  const int kx = PG == 4 ? (gq & 3) : gq;
  const bool yvalid = PG > 1 || gq + 8 < R;
  const int ky = PG == 1 ? (yvalid ? gq + 8 : gq) : kx;
  const uint32_t xo = xpage * ST + 4 * VB * (4 * kx + t4);
  const uint32_t yo = ypage * ST + 4 * VB * (4 * ky + t4);
  const uint32_t svxo = xpage * ST + OFF_S + var_sv_off(kx);
  const uint32_t svyo = ypage * ST + OFF_S + var_sv_off(ky);
  // coefficient words of product 2 (tokens gq and gq + 8)
  uint32_t co0 = 0, co1 = 0;
  if constexpr (PG == 4) {
    co0 = (t4 >> 1) * ST + OFF_C + 4 * (2 * gq + (t4 & 1));
    co1 = co0 + 2 * ST;
  } else if constexpr (PG == 2) {
    co0 = OFF_C + 4 * lane;
    co1 = co0 + ST;
  } else if constexpr (R == 15) {
    co0 = OFF_C + 32 * gq + 8 * t4;
  } else {
    co0 = OFF_C + (t4 < 2 ? 24 * gq + 8 * t4 : 24 * gq + 16 + 4 * (t4 - 2));
  }
  const uint32_t maskA = gq < 4 ? 0xffffffffu : 0u;      // MODE 1, PG 2
  const uint32_t maskP = (gq >> 2) == (t4 >> 1) ? 0xffffffffu : 0u;  // PG 4
  const uint32_t maskK = t4 < 2 ? 0xffffffffu : 0u;      // MODE 2/3, PG 4
  uint32_t bad = 0u;
#pragma unroll 1
  for (int g0 = 0; g0 < npg; g0 += PG) {
    const uint32_t gb = base_s + (uint32_t)g0 * ST;
    uint32_t xw[VC::words], yw[VC::words];
    load_slot<VB>(xw, gb + xo);
    load_slot<VB>(yw, gb + yo);
    const float svx = lds_f16(gb + svxo) * vscale;
    const float svy = yvalid ? lds_f16(gb + svyo) * vscale : 0.f;
    float d0[NT][4], d1[NT][4];
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      const uint32_t a[4] = {VC::op(xw, s, 0), VC::op(yw, s, 0),
                             VC::op(xw, s, 1), VC::op(yw, s, 1)};
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        if (s == 0)
          mma_f16_c(d0[nt], a, qv[nt][0][0], qv[nt][0][1], offc[nt][0],
                    offc[nt][1], offc[nt][0], offc[nt][1]);
        else if (s == 1)
          mma_f16_c(d1[nt], a, qv[nt][1][0], qv[nt][1][1], 0.f, 0.f, 0.f,
                    0.f);
        else if (s & 1)
          mma_f16(d1[nt], a, qv[nt][s][0], qv[nt][s][1]);
        else
          mma_f16(d0[nt], a, qv[nt][s][0], qv[nt][s][1]);
      }
    }
    // coefficient operands (exact codes): lo = token gq, hi = token gq + 8
    // (PG 1: b0/b1 = components 2t4.. / 8+2t4.. of a token)
    uint32_t c0lo, c0hi, c1lo = 0, c1hi = 0;
    if constexpr (PG > 1) {
      i8x4_to_h2(lds32(gb + co0), c0lo, c0hi);
      i8x4_to_h2(lds32(gb + co1), c1lo, c1hi);
    } else {
      uint32_t w0, w1;
      if (R == 15 || t4 < 2) {
        const uint2 u = lds64(gb + co0);
        w0 = u.x;
        w1 = u.y;
      } else {  // rank 12, components 4..7: both tokens in one word
        const uint32_t u = lds32(gb + co0);
        w0 = u;
        w1 = u >> 16;
      }
      i8x4_to_h2(w0, c0lo, c0hi);  // token gq
      i8x4_to_h2(w1, c1lo, c1hi);  // token gq + 8
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      // P (log2 units) split hi + lo, transposed per 8x8 block
      const float p0 = (d0[nt][0] + d1[nt][0]) * svx;
      const float p1 = (d0[nt][1] + d1[nt][1]) * svx;
      const float p2 = (d0[nt][2] + d1[nt][2]) * svy;
      const float p3 = (d0[nt][3] + d1[nt][3]) * svy;
      const __half2 hx = __floats2half2_rn(p0, p1);
      const __half2 hy = __floats2half2_rn(p2, p3);
      const uint32_t t0h = movmatrix_trans(h2_as_u32(hx));
      const uint32_t t0l = movmatrix_trans(split_lo(h2_as_u32(hx), p0, p1));
      const uint32_t t1h = movmatrix_trans(h2_as_u32(hy));
      const uint32_t t1l = movmatrix_trans(split_lo(h2_as_u32(hy), p2, p3));
      if constexpr (MODE == 1 && PG == 2) {
        // rows 0-3: page A heads, 4-7: page B heads (high), 8-15: low
        const uint32_t A2[4] = {t0h & maskA, t0l & maskA, t1h & ~maskA,
                                t1l & ~maskA};
        float l0[4], l1[4];
        mma_f16_z(l0, A2, c0lo, c1lo);
        mma_f16_z(l1, A2, c0hi, c1hi);
        const uint4 sc = lds128(gb + (gq < 4 ? 0 : ST) + OFF_S + 16 * t4);
        const float e = var_page_lse(l0, l1, sc.y, sc.z, SAFE, bad);
        if ((g0 >> 1) == t4) keep[0][0] = e;
      } else if constexpr (MODE == 1 && PG == 4) {
        // per block: rows 0-3 page 2 blk, rows 4-7 page 2 blk + 1
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {
          const uint32_t th = (blk ? t1h : t0h) & maskP;
          const uint32_t tl = (blk ? t1l : t0l) & maskP;
          float l0[4], l1[4];
          mma1688_f16_z(l0, th, tl, blk ? c1lo : c0lo);
          mma1688_f16_z(l1, th, tl, blk ? c1hi : c0hi);
          const uint4 sc =
              lds128(gb + (2 * blk + (gq >> 2)) * ST + OFF_S + 16 * t4);
          const float e = var_page_lse(l0, l1, sc.y, sc.z, SAFE, bad);
          if ((g0 >> 1) + blk == t4) keep[0][0] = e;
        }
      } else if constexpr (PG == 2) {
        float l0[4], l1[4];
        mma1688_f16_z(l0, t0h, t0l, c0lo);
        mma1688_f16_z(l1, t0h, t0l, c0hi);
        const uint4 sa = lds128(gb + OFF_S + 16 * t4);
        const float ea = var_page_lse(l0, l1, sa.y, sa.z, SAFE, bad);
        mma1688_f16_z(l0, t1h, t1l, c1lo);
        mma1688_f16_z(l1, t1h, t1l, c1hi);
        const uint4 sb = lds128(gb + ST + OFF_S + 16 * t4);
        const float eb = var_page_lse(l0, l1, sb.y, sb.z, SAFE, bad);
        if ((g0 >> 1) == t4) {
          keep[nt][0] = ea;
          keep[nt][1] = eb;
        }
      } else if constexpr (PG == 4) {
        // page 2 blk + u takes the K half of lanes t4 < 2 (u = 0) or
        // t4 >= 2 (u = 1) of block blk
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const uint32_t m = u ? ~maskK : maskK;
            float l0[4], l1[4];
            mma1688_f16_z(l0, blk ? t1h : t0h, blk ? t1l : t0l,
                          (blk ? c1lo : c0lo) & m);
            mma1688_f16_z(l1, blk ? t1h : t0h, blk ? t1l : t0l,
                          (blk ? c1hi : c0hi) & m);
            const uint4 sc = lds128(gb + (2 * blk + u) * ST + OFF_S + 16 * t4);
            const float e = var_page_lse(l0, l1, sc.y, sc.z, SAFE, bad);
            if ((g0 >> 1) + blk == t4) keep[nt][u] = e;
          }
        }
      } else {  // PG == 1: K 0..7 components 0..7, K 8..15 components 8..15
        const uint32_t A2[4] = {t0h, t0l, t1h, t1l};
        float l0[4], l1[4];
        mma_f16_z(l0, A2, c0lo, c0hi);
        mma_f16_z(l1, A2, c1lo, c1hi);
        const uint4 sc = lds128(gb + OFF_S + 16 * t4);
        const float e = var_page_lse(l0, l1, sc.y, sc.z, SAFE, bad);
        if ((g0 >> 1) == t4) keep[nt][g0 & 1] = e;
      }
    }
  }
  return bad;
}

// lane 0 starts the bulk copy of tile c (TP records of stride ST) into
// `dst`, completing on `bar`
template <int ST, int TP>
__device__ __forceinline__ void issue_var_tile(const Cursor &c,
                                               const int *nfull,
                                               const uint8_t *records,
                                               int h_kv, int max_pages,
                                               uint8_t *dst, uint64_t *bar,
                                               int lane) {
  if (lane == 0) {
    const int page0 = c.j * TP;
    const int npg = min(TP, nfull[c.b] - page0);
    const uint8_t *src =
        records + (((size_t)c.b * h_kv + c.h) * max_pages + page0) * (size_t)ST;
    const uint32_t bytes = (uint32_t)npg * ST;
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
    mbar_arrive_tx(bar, bytes);
    bulk_g2s(dst, src, bytes, bar);
  }
}

template <int R, int VB, int MODE>
__global__ void __launch_bounds__(32 * VarSched<R, VB>::W, 1)
    score_variant_kernel(const __nv_bfloat16 *__restrict__ q,
                         const uint8_t *__restrict__ records,
                         const int32_t *__restrict__ seq_lens, int batch,
                         int h_kv, int G, int max_pages,
                         float *__restrict__ s_hat, int32_t *status) {
  using S = VarSched<R, VB>;
  using VC = VCodes<VB>;
  constexpr int ST = S::stride, TP = S::TP, W = S::W, PG = var_pages_per_group(R);
  constexpr int NT = MODE == 3 ? 2 : 1;
  constexpr int OFF_MU = var_off_mu(R, VB), OFF_SMU = var_off_smu(R, VB);
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t *ring = smem;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S::ring);
  int *prefix = reinterpret_cast<int *>(bars + 2 * W);
  int *nfull = prefix + batch + 1;
  int *tph = nfull + batch;  // tiles per KV head of each sequence
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int gq = lane >> 2, t4 = lane & 3;
  const uint64_t keep_pol = l2_keep_policy();

  for (int b = threadIdx.x; b < batch; b += blockDim.x) {
    int L = seq_lens[b];
    if (L < 0 || L > max_pages * kPage) {
      if (blockIdx.x == 0) set_status(status, LOCKS_DEV_BAD_SEQ_LEN);
      L = max(0, min(L, max_pages * kPage));
    }
    nfull[b] = L / kPage;
    tph[b] = (L / kPage + TP - 1) / TP;
    prefix[b + 1] = tph[b] * h_kv;
  }
  if (threadIdx.x == 0) prefix[0] = 0;
  if (lane == 0) {
    mbar_init(&bars[2 * wid], 1);
    mbar_init(&bars[2 * wid + 1], 1);
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
  const long long nw = (long long)gridDim.x * W;
  const long long gw = (long long)blockIdx.x * W + wid;
  const long long t_begin = gw * total / nw, t_end = (gw + 1) * total / nw;
  if (t_begin >= t_end) return;
  uint8_t *my_ring = ring + (size_t)wid * 2 * S::tile;
  const uint32_t ring_s = smem_u32(my_ring);
  uint64_t *my_bar = bars + 2 * wid;

  Cursor cur{0, 0, 0};
  {  // largest b with prefix[b] <= t_begin
    int lo = 0, hi = batch;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (prefix[mid] <= t_begin) lo = mid; else hi = mid;
    }
    const int rem = (int)(t_begin - prefix[lo]);
    cur.b = lo;
    cur.h = rem / tph[lo];
    cur.j = rem - cur.h * tph[lo];
  }
  Cursor nxt = cur;
  issue_var_tile<ST, TP>(nxt, nfull, records, h_kv, max_pages, my_ring,
                         &my_bar[0], lane);
  advance_cursor(nxt, tph, batch, h_kv);
  if (t_begin + 1 < t_end) {
    issue_var_tile<ST, TP>(nxt, nfull, records, h_kv, max_pages,
                           my_ring + S::tile, &my_bar[1], lane);
    advance_cursor(nxt, tph, batch, h_kv);
  }

  uint32_t qv[NT][8][2];  // product-1 B fragments (divided by the scales)
  float offc[NT][2];      // code offsets of columns 2 t4, 2 t4 + 1
  uint32_t qh[8][4];      // product-3 A fragments (heads gq, gq + 8)
  float off_m = 0.f, off_m8 = 0.f;
  float vscale = kLog2eRsqrtD;
  int cur_b = -1, cur_h = -1;
  bool failed = false;
  float *unit_rows = nullptr;
  const int n_tiles = (int)(t_end - t_begin);

  for (int it = 0; it < n_tiles; ++it) {
    const int stage = it & 1;
    const uint32_t phase = (uint32_t)((it >> 1) & 1);
    if (cur.b != cur_b || cur.h != cur_h) {
      cur_b = cur.b;
      cur_h = cur.h;
      unit_rows =
          s_hat + ((size_t)cur.b * h_kv + cur.h) * G * (size_t)max_pages;
      const __nv_bfloat16 *qrow =
          q + ((size_t)cur.b * h_kv * G + (size_t)cur.h * G) * kDim;
      // power-of-two prescale bringing max |q| of the group into
      // [2^13, 2^14): every fp16 operand (also q / 256 of 2-bit codes)
      // stays normal down to 2^-19 of the largest element
      float amax = 0.f;
      uint32_t qb[8][4];
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const int d0 = 16 * s + 2 * t4;
        uint32_t u0 = 0, u1 = 0, u2 = 0, u3 = 0;
        if (gq < G) {
          u0 = __ldg(reinterpret_cast<const uint32_t *>(qrow + gq * kDim + d0));
          u2 = __ldg(reinterpret_cast<const uint32_t *>(qrow + gq * kDim + d0 + 8));
        }
        if (gq + 8 < G) {
          u1 = __ldg(reinterpret_cast<const uint32_t *>(qrow + (gq + 8) * kDim + d0));
          u3 = __ldg(reinterpret_cast<const uint32_t *>(qrow + (gq + 8) * kDim + d0 + 8));
        }
        qb[s][0] = u0;
        qb[s][1] = u1;
        qb[s][2] = u2;
        qb[s][3] = u3;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(qb[s][i])),
                                   fabsf(bf16_hi(qb[s][i]))));
      }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      int ex = 0;
      if (amax > 0.f && amax < INFINITY)
        ex = min(125, max(-125, ((__float_as_int(amax) >> 23) & 0xff) - 140));
      const float qsc = __int_as_float((127 - ex) << 23);  // 2^-ex
      vscale = kLog2eRsqrtD * __int_as_float((127 + ex) << 23);
      float sumh = 0.f, sumh8 = 0.f;
#pragma unroll
      for (int s = 0; s < 8; ++s) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t u = qb[s][i];
          const __half2 hq =
              __floats2half2_rn(bf16_lo(u) * qsc, bf16_hi(u) * qsc);
          qh[s][i] = h2_as_u32(hq);
          if (i & 1)
            sumh8 += __low2float(hq) + __high2float(hq);
          else
            sumh += __low2float(hq) + __high2float(hq);
        }
      }
      sumh += __shfl_xor_sync(0xffffffffu, sumh, 1);
      sumh += __shfl_xor_sync(0xffffffffu, sumh, 2);
      sumh8 += __shfl_xor_sync(0xffffffffu, sumh8, 1);
      sumh8 += __shfl_xor_sync(0xffffffffu, sumh8, 2);
      off_m = -1152.f * sumh;  // cancels the +1152 of every centroid code
      off_m8 = -1152.f * sumh8;
      // product 1's columns: head (n mod 4) for MODE 1, else head n + 8 nt
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int hc = MODE == 1 ? (gq & 3) : gq + 8 * nt;
        const __nv_bfloat16 *qc = qrow + hc * kDim;
        float cs = 0.f;
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          const int d0 = 16 * s + 2 * t4;
          const uint32_t u =
              hc < G ? __ldg(reinterpret_cast<const uint32_t *>(qc + d0)) : 0u;
          const uint32_t u8 =
              hc < G ? __ldg(reinterpret_cast<const uint32_t *>(qc + d0 + 8))
                     : 0u;
          const float f0 = qsc / VC::scale(s, 0), f1 = qsc / VC::scale(s, 1);
          const __half2 lo = __floats2half2_rn(bf16_lo(u) * f0, bf16_hi(u) * f0);
          const __half2 hi =
              __floats2half2_rn(bf16_lo(u8) * f1, bf16_hi(u8) * f1);
          qv[nt][s][0] = h2_as_u32(lo);
          qv[nt][s][1] = h2_as_u32(hi);
          cs -= VC::offset(s, 0) * (__low2float(lo) + __high2float(lo)) +
                VC::offset(s, 1) * (__low2float(hi) + __high2float(hi));
        }
        cs += __shfl_xor_sync(0xffffffffu, cs, 1);
        cs += __shfl_xor_sync(0xffffffffu, cs, 2);
        offc[nt][0] = __shfl_sync(0xffffffffu, cs, 4 * (2 * t4));
        offc[nt][1] = __shfl_sync(0xffffffffu, cs, 4 * (2 * t4 + 1));
      }
    }
    const int page0 = cur.j * TP;
    const int npg = min(TP, nfull[cur.b] - page0);
    if (!mbar_wait(&my_bar[stage], phase)) {
      failed = true;
      break;
    }
    const uint32_t base_s = ring_s + stage * S::tile;
    // the rest of a partial last group is zeroed (a zero record scores to a
    // finite constant), so what the ring held before takes no part in the
    // overflow vote
    if (PG > 1 && npg % PG) {
      const int pad = PG - npg % PG;
      uint4 *slot =
          reinterpret_cast<uint4 *>(my_ring + stage * S::tile + npg * ST);
      for (int i = lane; i < pad * ST / 16; i += 32)
        slot[i] = make_uint4(0u, 0u, 0u, 0u);
      __syncwarp();
    }
    float keep[NT][2] = {};
    const uint32_t bad = var_score_groups<R, VB, MODE, false>(
        base_s, npg, lane, qv, offc, vscale, keep);
    if (__any_sync(0xffffffffu, bad >= kLseBad))
      var_score_groups<R, VB, MODE, true>(base_s, npg, lane, qv, offc, vscale,
                                          keep);
    // q . mu for the tile's pages (column n = page n of the tile; with 4-page
    // tiles columns 4..7 repeat pages 0..3)
    float qm[4] = {off_m, off_m, off_m8, off_m8};
    float qm2[4] = {0.f, 0.f, 0.f, 0.f};
    {
      const uint32_t mrow = base_s + (gq & (TP - 1)) * ST + OFF_MU + 32 * t4;
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
    const float mscale = vscale;
    if constexpr (MODE == 1) {
      // lane (g, t4) of the low half: page 2 t4; of the high half: page
      // 2 t4 + 1; head g & 3
      const bool up = gq >= 4;
      const float qm_hi_lane = __shfl_xor_sync(0xffffffffu, qm[1] + qm2[1], 16);
      const int pg = 2 * t4 + (up ? 1 : 0), head = gq & 3;
      const float qmu = up ? qm_hi_lane : qm[0] + qm2[0];
      if (head < G && pg < npg) {
        const float smu = lds_f16(base_s + pg * ST + OFF_SMU);
        st_keep(unit_rows + (size_t)head * max_pages + page0 + pg,
                (keep[0][0] + qmu * smu * mscale) * kLn2, keep_pol);
      }
    } else {
      const int pg0 = 2 * t4, pg1 = pg0 + 1;
      const float sm0 = pg0 < npg ? lds_f16(base_s + pg0 * ST + OFF_SMU) : 0.f;
      const float sm1 = pg1 < npg ? lds_f16(base_s + pg1 * ST + OFF_SMU) : 0.f;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int head = gq + 8 * nt;
        if (head < G) {
          float *dst = unit_rows + (size_t)head * max_pages + page0;
          if (pg0 < npg)
            st_keep(dst + pg0,
                    (keep[nt][0] + (qm[2 * nt] + qm2[2 * nt]) * sm0 * mscale) *
                        kLn2,
                    keep_pol);
          if (pg1 < npg)
            st_keep(dst + pg1,
                    (keep[nt][1] +
                     (qm[2 * nt + 1] + qm2[2 * nt + 1]) * sm1 * mscale) *
                        kLn2,
                    keep_pol);
        }
      }
    }
    __syncwarp();
    if (it + 2 < n_tiles) {
      issue_var_tile<ST, TP>(nxt, nfull, records, h_kv, max_pages,
                             my_ring + stage * S::tile, &my_bar[stage], lane);
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
}

template <int R, int VB, int MODE>
cudaError_t launch_variant_mode(const void *q, const void *records,
                                const int32_t *seq_lens, int batch, int h_kv,
                                int G, int max_pages, float *scores,
                                int32_t *status, cudaStream_t stream) {
  const size_t smem = variant_smem_bytes<R, VB>(batch);
  cudaError_t e = cudaFuncSetAttribute(
      score_variant_kernel<R, VB, MODE>,
      cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  score_variant_kernel<R, VB, MODE>
      <<<device_sm_count(), 32 * VarSched<R, VB>::W, smem, stream>>>(
          static_cast<const __nv_bfloat16 *>(q),
          static_cast<const uint8_t *>(records), seq_lens, batch, h_kv, G,
          max_pages, scores, status);
  return launched();
}

template <int R, int VB>
cudaError_t launch_variant_rv(const void *q, const void *records,
                              const int32_t *seq_lens, int batch, int h_kv,
                              int G, int max_pages, float *scores,
                              int32_t *status, cudaStream_t stream) {
  if (G > 8)
    return launch_variant_mode<R, VB, 3>(q, records, seq_lens, batch, h_kv, G,
                                         max_pages, scores, status, stream);
  if constexpr (var_pages_per_group(R) > 1) {
    if (G <= 4)
      return launch_variant_mode<R, VB, 1>(q, records, seq_lens, batch, h_kv,
                                           G, max_pages, scores, status,
                                           stream);
  }
  return launch_variant_mode<R, VB, 2>(q, records, seq_lens, batch, h_kv, G,
                                       max_pages, scores, status, stream);
}

// one translation unit per basis width instantiates its four ranks
template <int VB>
cudaError_t launch_variant_bits(int rank, const void *q, const void *records,
                                const int32_t *seq_lens, int batch, int h_kv,
                                int G, int max_pages, float *scores,
                                int32_t *status, cudaStream_t stream) {
  switch (rank) {
    case 4:
      return launch_variant_rv<4, VB>(q, records, seq_lens, batch, h_kv, G,
                                      max_pages, scores, status, stream);
    case 8:
      return launch_variant_rv<8, VB>(q, records, seq_lens, batch, h_kv, G,
                                      max_pages, scores, status, stream);
    case 12:
      return launch_variant_rv<12, VB>(q, records, seq_lens, batch, h_kv, G,
                                       max_pages, scores, status, stream);
    case 15:
      return launch_variant_rv<15, VB>(q, records, seq_lens, batch, h_kv, G,
                                       max_pages, scores, status, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace locks
