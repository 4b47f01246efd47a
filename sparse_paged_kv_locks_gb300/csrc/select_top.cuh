// Radix select and ordered compaction of one (sequence, KV head)'s
// candidate keys (LOCKS reading notes §4.2, the sink/recent rule: the
// sink page, the recent page and the k-2 candidate pages of largest key,
// ties to the lower page, ascending), shared by the selection kernel and
// the fused score-and-select kernel.  Included by those .cu files only.
#pragma once

#include "common.cuh"

namespace locks {

constexpr int kSelThreads = 512;

// Keys are order keys of the float key (monotone as unsigned integers);
// the sink, the recent page and pages past the candidates hold key 0,
// which is below every real key.
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

// Radix digits: 12 bits, scanned 256 digits per warp of the 512-thread
// block.
constexpr int kRadixBits = 12;
constexpr int kRadixBins = 1 << kRadixBits;
constexpr int kBinsPerWarp = kRadixBins / (kSelThreads / 32);  // 256


// Shared-memory scratch of select_top.
struct SelectScratch {
  int hist[2][kRadixBins];
  int wcnt[2][32];
  uint32_t prefix, mask;
  int remaining, varying;
};

// The k-2 candidates of largest key among keys[0..n) (n > k >= 3, at least
// k-2 candidates) by radix select over the bits where the candidate keys
// differ (kmin, kmax: their minimum and maximum, read by thread 0), then
// out[0] = 0 (sink), out[1..k-2] the selected pages ascending, out[k-1] =
// n-1 (recent).  Called by every thread of a 512-thread block; `kvec`:
// keys 16-byte aligned in groups of four; s.hist[0] must be zero on entry
// (the caller clears it while other work runs).
template <bool SMEM_KEYS, int NWARPS>
__device__ __forceinline__ void select_top(const uint32_t *keys, bool kvec,
                                           int n, int k, uint32_t kmin,
                                           uint32_t kmax, int32_t *out,
                                           int32_t *status,
                                           SelectScratch &s) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  if (tid == 0) {
    const uint32_t a = kmin, z = kmax;
    // bits above the highest one where min and max differ are common to
    // every candidate key
    const int varying = (a == z) ? 0 : 32 - __clz(a ^ z);
    const uint32_t msk = varying == 32 ? 0u : ~((1u << varying) - 1u);
    s.prefix = z & msk;
    s.mask = msk;
    s.remaining = k - 2;
    s.varying = varying;
  }
  __syncthreads();

  // radix select of the (k-2)-th largest key over the varying bits,
  // 12-bit digits from the top; key 0 never matches a candidate prefix.
  // Histograms alternate between two buffers so the next one is cleared
  // while the current one fills.
  const int varying = s.varying;
  const int nk4 = (n + 3) >> 2;
  for (int top = varying, pass = 0; top > 0; top -= kRadixBits, ++pass) {
    const int width = min(kRadixBits, top), shift = top - width;
    const uint32_t dmask = (1u << width) - 1u;
    int *hc = s.hist[pass & 1];
    int *hn = s.hist[(pass & 1) ^ 1];
    const uint32_t pre = s.prefix, msk = s.mask;
    const int rem = s.remaining;
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
    if (lane == 31) s.wcnt[0][wid] = incl;
    __syncthreads();
    const int before = warps_before<NWARPS>(s.wcnt[0], wid, lane);
    const int mine = before + incl - cnt;  // count above this lane's digits
    if (mine < rem && rem <= mine + cnt) {
      const int c[8] = {c4.w, c4.z, c4.y, c4.x,
                        d4.w, d4.z, d4.y, d4.x};  // digits hi, hi-1, ...
      int acc = mine;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (acc < rem && rem <= acc + c[i]) {
          s.prefix = pre | ((uint32_t)(hi - i) << shift);
          s.mask = msk | (dmask << shift);
          s.remaining = rem - acc;
        }
        acc += c[i];
      }
    }
    __syncthreads();
  }
  const uint32_t T = s.prefix;
  const int need_eq = s.remaining;  // keys equal to T to keep (lowest j)

  // ordered compaction: warp w owns pages [w*seg, (w+1)*seg), walked 128 at
  // a time (four per lane); warps' counts are scanned once
  const int seg = ((n + NWARPS - 1) / NWARPS + 127) & ~127;
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
    if (lane == 0) s.wcnt[0][wid] = (eq << 16) | gt;
    __syncthreads();
    const int ge_before = warps_before<NWARPS>(s.wcnt[0], wid, lane);
    gt_before = ge_before & 0xffff;
    eq_before = ge_before >> 16;
  } else {
    if (lane == 0) {
      s.wcnt[0][wid] = gt;
      s.wcnt[1][wid] = eq;
    }
    __syncthreads();
    gt_before = warps_before<NWARPS>(s.wcnt[0], wid, lane);
    eq_before = warps_before<NWARPS>(s.wcnt[1], wid, lane);
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

}  // namespace locks
