// GQA-shared page selection (LOCKS reading notes §4.2 Eq.(5) with the
// sink/recent rule, §4.4 Algorithm 2): per (sequence, KV head), normalise
// each head's page scores into mass fractions, average them over the group
// and keep the sink page, the recent page and the k-2 other pages of largest
// share (ties to the lower page).
#include "common.cuh"
#include "launch.h"
#include "select_top.cuh"

namespace locks {

// ---------------------------------------------------------------------------
// selection: one CTA per (sequence, KV head)
// ---------------------------------------------------------------------------
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

// Keys live in shared memory when they fit (SMEM_KEYS), else in the
// workspace.  Keys are indexed by page; the sink, the recent page and pages
// past the candidates hold key 0, which is below every real key.
// MINB: resident CTAs per SM the registers are sized for.  2 when there are
// more (sequence, KV head) units than SMs; 1 when every unit has an SM of
// its own, which leaves registers for more pages in flight per thread.
// CL > 1: a thread-block cluster of CL CTAs per unit (few units): each CTA
// takes 1/CL of the unit's pages through the normaliser and key passes, the
// per-head sums are merged through distributed shared memory in rank order
// (the same Z_g in every CTA), the keys go to CTA 0's shared memory and
// CTA 0 selects.
template <bool SMEM_KEYS, int GT, int MINB, int CL = 1>
__global__ void __launch_bounds__(kSelThreads, MINB)
    select_kernel(const float *__restrict__ scores,
                  const int32_t *__restrict__ seq_lens, int h_kv, int G,
                  int max_pages, int k, int rule,
                  int32_t *__restrict__ idx, uint32_t *__restrict__ keybuf,
                  int32_t *status) {
  extern __shared__ __align__(16) uint32_t sel_keys[];
  __shared__ float zs[kMaxGroup];
  __shared__ float red_m[32][kMaxGroup], red_s[32][kMaxGroup];
  __shared__ __align__(16) SelectScratch sel;
  __shared__ uint32_t red_u[2][32];
  __shared__ int sh_slow;
  // CL > 1: this CTA's per-head sums (fast and general normaliser forms)
  // and, in CTA 0, every rank's (kmin, kmax)
  __shared__ float c_s[kMaxGroup], c_m2[kMaxGroup], c_s2[kMaxGroup];
  __shared__ uint32_t c_kmm[2][CL];
  static_assert(!(CL > 1) || SMEM_KEYS, "clusters keep the keys on chip");

  const int rank = CL > 1 ? (int)cluster_ctarank() : 0;
  const int b = blockIdx.y, h = CL > 1 ? (int)blockIdx.x / CL : blockIdx.x;
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
    if (rank == 0)
      for (int i = tid; i < k; i += blockDim.x) out[i] = i < n ? i : -1;
    return;
  }
  if (k == 2) {  // only the sink and the recent page
    if (tid == 0 && rank == 0) {
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
  // this CTA's quads [qa, qb) (the whole unit when CL = 1)
  const int qper = (nq + CL - 1) / CL;
  const int qa = min(nq, rank * qper), qb = min(nq, qa + qper);
  const int nlim = min(nf, 4 * qb);   // summarised pages of this CTA's range
  // quads a thread has in flight at once (what the registers allow)
  // (at two CTAs per SM and G = 4 a second quad in flight measured slower,
  // 16.6 against 16.2 us on 256 units, and spilled)
  constexpr int R = MINB == 1 ? (GT <= 8 ? 2 : 1) : (GT <= 2 ? 2 : 1);
  for (int i = tid; i < kRadixBins; i += blockDim.x) sel.hist[0][i] = 0;

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
    for (int qd = qa + tid; qd < qb; qd += R * blockDim.x) {
      float x[R][GT][4];
#pragma unroll
      for (int r = 0; r < R; ++r)
        load_quad<GT>(sc, max_pages, G, vec, 4 * (qd + r * blockDim.x), nlim,
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
    float sum = 0.f;
    if (tid < G)
      for (int w = 0; w < nwarps; ++w) sum += red_s[w][tid];
    if constexpr (CL > 1) {  // the cluster's sums, in rank order
      if (tid < G) c_s[tid] = sum;
      cluster_sync();
      if (tid < G) {
        sum = 0.f;
        for (int c = 0; c < CL; ++c)
          sum += ld_cluster_f32(mapa_shared(smem_u32(&c_s[tid]), c));
      }
    }
    if (tid < G) {
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
    for (int qd = qa + tid; qd < qb; qd += R * blockDim.x) {
      float x[R][GT][4];
#pragma unroll
      for (int r = 0; r < R; ++r)
        load_quad<GT>(sc, max_pages, G, vec, 4 * (qd + r * blockDim.x), nlim,
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
  float m = -INFINITY, s = 0.f;
  if (tid < G) {
    for (int w = 0; w < nwarps; ++w) m = fmaxf(m, red_m[w][tid]);
    for (int w = 0; w < nwarps; ++w)
      if (red_m[w][tid] != -INFINITY)
        s += red_s[w][tid] * ex2_fast(red_m[w][tid] - m);
  }
  if constexpr (CL > 1) {  // the cluster's (m, s) pairs, in rank order
    if (tid < G) {
      c_m2[tid] = m;
      c_s2[tid] = s;
    }
    cluster_sync();
    if (tid < G) {
      m = -INFINITY;
      s = 0.f;
      for (int c = 0; c < CL; ++c) {
        const float m2 = ld_cluster_f32(mapa_shared(smem_u32(&c_m2[tid]), c));
        const float s2 = ld_cluster_f32(mapa_shared(smem_u32(&c_s2[tid]), c));
        const float mm = fmaxf(m, m2);
        if (mm == -INFINITY) continue;
        s = (m == -INFINITY ? 0.f : s * ex2_fast(m - mm)) +
            (m2 == -INFINITY ? 0.f : s2 * ex2_fast(m2 - mm));
        m = mm;
      }
    }
  }
  if (tid < G) zs[tid] = m + lg2_fast(s);
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
  for (int it = (qb - qa + qstep - 1) / qstep - 1; it >= 0; --it) {
    const int qd = qa + it * qstep + tid;
    if (qd >= qb) continue;
    float x[R][GT][4];
    // heads at or above G read -inf: no term, no maximum
#pragma unroll
    for (int r = 0; r < R; ++r)
      load_quad<GT>(sc, max_pages, G, vec, 4 * (qd + r * blockDim.x), nf,
                    -INFINITY, x[r]);
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int j0 = 4 * (qd + r * blockDim.x);
      if (j0 >= 4 * qb) break;
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
      if (CL > 1) {  // into CTA 0's key array
        st_cluster_v4(mapa_shared(smem_u32(keys + j0), 0),
                      make_uint4(kq[0], kq[1], kq[2], kq[3]));
      } else if (kvec) {
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
  uint32_t a = 0xffffffffu, z = 0u;
  if (tid == 0) {
    for (int w = 0; w < nwarps; ++w) {
      a = min(a, red_u[0][w]);
      z = max(z, red_u[1][w]);
    }
  }
  if constexpr (CL > 1) {
    if (tid == 0) {
      st_cluster_u32(mapa_shared(smem_u32(&c_kmm[0][rank]), 0), a);
      st_cluster_u32(mapa_shared(smem_u32(&c_kmm[1][rank]), 0), z);
    }
    cluster_sync();  // CTA 0 holds every key and every rank's bounds
    if (rank != 0) return;
    if (tid == 0)
      for (int c = 0; c < CL; ++c) {
        a = min(a, c_kmm[0][c]);
        z = max(z, c_kmm[1][c]);
      }
  }
  select_top<SMEM_KEYS, nwarps>(keys, kvec, n, k, a, z, out, status, sel);
}

// --------------------------------------------------------------------------
// launcher
// --------------------------------------------------------------------------
constexpr int kSelSmemKeys = 32 * 1024;   // candidate keys held on chip

// CTAs per (sequence, KV head) unit: 4 or 2 when that many clusters fit the
// SMs in one wave and the lists are long, else 1.  Measured on GB300 (graph
// replay): 64 units of 8,208 pages at G = 8, 15.6 -> 14.0 us with clusters
// of 2; 64 units of 2,048 pages at G = 4, 7.4 -> 8.2 us (the cluster
// barriers and the remote key stores cost more than the halved passes save),
// hence the 4,096-page floor.
constexpr int kSelClusterMinPages = 4096;

int select_cluster_size(long long units, int max_pages) {
  const int sms = device_sm_count();
  if (max_pages < kSelClusterMinPages) return 1;
  if (units * 4 <= sms) return 4;
  if (units * 2 <= sms) return 2;
  return 1;
}

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
  const long long units = (long long)batch * h_kv;
  const bool own_sm = units <= device_sm_count();
  // with few units, a cluster of CTAs per unit shares its passes
  const int cl = on_chip ? select_cluster_size(units, max_pages) : 1;
  if (cl > 1) {
    auto run_cl = [&](auto kern) -> cudaError_t {
      cudaError_t e = cudaFuncSetAttribute(
          kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSelSmemKeys * 4);
      if (e != cudaSuccess) return e;
      return launch_pdl_cluster(kern, dim3(h_kv * cl, batch),
                                dim3(kSelThreads), smem, stream, cl, scores,
                                seq_lens, h_kv, G, max_pages, k, rule, idx,
                                keybuf, status);
    };
#define LOCKS_SELECT_CL(C)                                   \
  switch (gt) {                                              \
    case 1: return run_cl(select_kernel<true, 1, 1, C>);     \
    case 2: return run_cl(select_kernel<true, 2, 1, C>);     \
    case 4: return run_cl(select_kernel<true, 4, 1, C>);     \
    case 8: return run_cl(select_kernel<true, 8, 1, C>);     \
    default: return run_cl(select_kernel<true, 16, 1, C>);   \
  }
    if (cl == 4) LOCKS_SELECT_CL(4)
    LOCKS_SELECT_CL(2)
#undef LOCKS_SELECT_CL
  }
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
