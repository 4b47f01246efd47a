// Byte layout of the rank / precision variant records (LOCKS reading notes
// §6, the ablation on rank and quantisation precision; include/locks.h has
// the normative description).  The layout follows the shipped record's
// rule -- every scoring lane finds its tensor-core fragments in one or two
// aligned shared-memory words -- generalised to rank R in {4, 8, 12, 15}
// and a basis of VB in {2, 4, 8} bits; the (8, 4) record is byte for byte
// the shipped 832-byte record.
//
// Product 1 of the scorer is the transposed basis product: mma rows are
// basis components of PG pages (PG = 4 for R = 4, 2 for R = 8, 1 for R = 12
// and 15), so a lane (gq = lane / 4, t = lane % 4) needs, for one component
// k, the 32 codes of head dims d = 16 s + 2 t + e + 8 h (s < 8, e, h < 2):
// the "slot" (k, t), 4 VB bytes at 4 VB (4 k + t).  Inside a slot:
//   VB = 4: word s/2, bits 16 e + 8 (s%2) + 4 h, two's complement nibbles
//   VB = 2: word s/4, bits 16 e + 2 (2 (s%4) + h), two's complement
//   VB = 8: byte 4 s + 2 h + e, stored excess-128
// Coefficient codes C[i][k] (excess-128) are ordered by the lane that feeds
// them to product 2, the centroid codes as in the shipped record, and the
// fp16 scales sit in the shipped 64-byte scale block (sV[2t], sV[2t+1],
// sC[2t], sC[2t+1], sC[8+2t], sC[9+2t] in group t; for R > 8 the group's
// last four bytes hold sV[8+2t], sV[9+2t] and sMU takes the sV[15] slot).
#pragma once
#include <stddef.h>

#include "common.cuh"

namespace locks {

__host__ __device__ constexpr int var_pages_per_group(int r) {
  return r == 4 ? 4 : r == 8 ? 2 : 1;
}
__host__ __device__ constexpr int var_coeff_bytes(int r) {
  return r <= 8 ? 16 * r : r == 12 ? 192 : 256;
}
__host__ __device__ constexpr int var_off_c(int r, int vbits) {
  return 16 * r * vbits;
}
__host__ __device__ constexpr int var_off_mu(int r, int vbits) {
  return var_off_c(r, vbits) + var_coeff_bytes(r);
}
__host__ __device__ constexpr int var_off_s(int r, int vbits) {
  return var_off_mu(r, vbits) + kDim;
}
__host__ __device__ constexpr int var_off_smu(int r, int vbits) {
  return var_off_s(r, vbits) + (r <= 8 ? 12 : 62);
}
__host__ __device__ constexpr int var_stride(int r, int vbits) {
  return var_off_s(r, vbits) + 64;
}

// byte offset, inside the scale block, of the basis scale sV[k]
__host__ __device__ constexpr int var_sv_off(int k) {
  return k < 8 ? 16 * (k >> 1) + 2 * (k & 1)
               : 16 * ((k - 8) >> 1) + 12 + 2 * (k & 1);
}
// ... of the coefficient scale sC[i]
__host__ __device__ constexpr int var_sc_off(int i) {
  return 16 * ((i & 7) >> 1) + 4 + 2 * (i & 1) + 4 * (i >> 3);
}

// byte offset, inside the coefficient region, of C[i][k] (k < r)
__host__ __device__ constexpr int var_c_off(int r, int i, int k) {
  const int g = i & 7, hi = i >> 3;
  if (r <= 8) return 4 * (g * (r / 2) + k / 2) + 2 * hi + (k & 1);
  const int t = (k & 7) >> 1;  // the lane (g, t) that reads it
  if (r == 12 && t >= 2) return 24 * g + 16 + 4 * (t - 2) + 2 * hi + (k & 1);
  const int per = r == 12 ? 24 : 32;
  return per * g + 8 * t + 4 * hi + 2 * (k >> 3) + (k & 1);
}

// byte offset, inside the basis region, of the code of V[d][k], and the bit
// of that byte where it starts
__host__ __device__ constexpr int var_v_bit(int vbits, int d, int k) {
  const int t = (d & 7) >> 1, e = d & 1, h = (d & 15) >> 3, s = d >> 4;
  const int slot_bits = 32 * vbits * (4 * k + t);
  if (vbits == 4) return slot_bits + 32 * (s >> 1) + 16 * e + 8 * (s & 1) + 4 * h;
  if (vbits == 2) return slot_bits + 32 * (s >> 2) + 16 * e + 2 * (2 * (s & 3) + h);
  return slot_bits + 8 * (4 * s + 2 * h + e);
}

// byte offset, inside the centroid region, of mu[d] (the shipped order)
__host__ __device__ constexpr int var_mu_off(int d) {
  return 32 * ((d & 7) >> 1) + 4 * (d >> 4) + (d & 1) + 2 * ((d & 15) >> 3);
}

// scorer tiling (variant_score.cuh): tile pages, warps per CTA, ring bytes
// shared-memory ring of every variant's scorer (the shipped scorer's)
constexpr int kVarRingMax = 212992;

template <int R, int VB>
struct VarSched {
  static constexpr int stride = var_stride(R, VB);
  // tile pages: 8 when sixteen warps' double-buffered tiles fit the ring
  static constexpr int TP = 16 * 2 * 8 * stride <= kVarRingMax ? 8 : 4;
  static constexpr int tile = TP * stride;
  static constexpr int W =
      kVarRingMax / (2 * tile) > 16 ? 16 : kVarRingMax / (2 * tile);
  static constexpr int ring = W * 2 * tile;
  static_assert(W >= 4, "at least four warps per CTA");
};

template <int R, int VB>
size_t variant_smem_bytes(int batch) {
  using S = VarSched<R, VB>;
  return (size_t)S::ring + 2 * sizeof(uint64_t) * S::W +
         sizeof(int) * (3 * (size_t)batch + 1);
}

}  // namespace locks
