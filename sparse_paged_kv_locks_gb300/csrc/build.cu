// Page summary build (LOCKS reading notes §4.1 Eq.(2)-(3), §4.3 Algorithm 1),
// summary packing and append-with-incremental-build.
//
// One warp per (page, KV head).  Lane l owns head dims 4l..4l+3 of all 16
// tokens, so centring, the basis V = D^T U_r Sigma_r^{-1} and the
// quantisation of the centroid are lane-local.  The 16x16 Gram matrix is
// accumulated as per-lane partials and reduce-scattered across the warp; the
// symmetric eigenproblem runs as a cyclic two-sided Jacobi iteration with the
// round-robin (circle) ordering, eight disjoint rotations per round.  The
// matrix and the eigenvector accumulator live in shared memory in "slot"
// order: slots 2m and 2m+1 always hold the two indices that round's pair m
// rotates, and each round writes its result to the other buffer with the
// slots moved for the next round (a fixed permutation, so every address a
// lane touches is a constant).  A lane rotates two 2x2 blocks of the matrix
// and, in registers, its own pair's two eigenvector columns over four rows,
// which then move to the next round's slots by two neighbour shuffles; one
// warp barrier per round.
#include <utility>

#include "common.cuh"
#include "launch.h"
#include "variant_layout.cuh"

namespace locks {

constexpr int kBuildWarps = 4;
constexpr int kMaxSweeps = 15;
constexpr float kJacobiRelTol = 1e-7f;
constexpr int kAS = 24;  // row stride (floats) of the Jacobi matrix copy

// 16-byte aligned so that every warp's copy keeps the float2 accesses of
// the eigensolve aligned
struct alignas(16) BuildSmem {
  union {
    struct {  // the eigensolve: slot order, double-buffered
      float Ab[2][16][kAS];
    } jac;
    struct {  // after it
      float U[16][17];  // eigenvectors (columns), index order
      float Cf[16][8];
      int8_t v8[128][8];
      int8_t c8[16][8];
      int8_t m8[128];
    } post;
  };
  float ev[16];  // eigenvalues, index order
  float lam[16];
  int perm[16];
  float cv[8], cc[8];
  __half sv[8], sc[16], smu;
};
// the append kernel keeps one per KV head (up to 32) in one CTA
static_assert(32 * sizeof(BuildSmem) <= 227 * 1024, "append smem");
static_assert(sizeof(BuildSmem) % 16 == 0, "per-warp copies stay aligned");

// Round-robin slots.  At round 0 of every sweep slot 2m holds index p_m and
// slot 2m+1 index q_m of pair m (p_0 = 0, p_m = m, q_m = 15 - m); after a
// round the index in slot a moves to slot slot_next(a).  Fifteen rounds
// bring every index back, so sweeps start and end in this arrangement.
__host__ __device__ constexpr int slot_index(int a) {
  return a == 0 ? 0 : (a & 1) ? 15 - (a - 1) / 2 : a / 2;
}
__host__ __device__ constexpr int index_slot(int i) {
  return i == 0 ? 0 : i <= 7 ? 2 * i : 2 * (15 - i) + 1;
}
__host__ __device__ constexpr int slot_next(int a) {
  return a == 0 ? 0 : a == 2 ? 1 : a == 15 ? 14 : (a & 1) ? a + 2 : a - 2;
}
// Upper-triangle pair (i <= j) enumeration of the 16x16 Gram matrix.
__host__ __device__ constexpr int pair_i(int p) {
  int i = 0;
  while (i < 16 && p >= 16 - i) {
    p -= 16 - i;
    ++i;
  }
  return i;
}
__host__ __device__ constexpr int pair_j(int p) {
  int i = 0;
  while (i < 16 && p >= 16 - i) {
    p -= 16 - i;
    ++i;
  }
  return i + p;
}

template <int P>
__device__ __forceinline__ float gram_partial(const float (&D)[16][4]) {
  if constexpr (P >= 136) {
    return 0.f;
  } else {
    constexpr int i = pair_i(P), j = pair_j(P);
    return D[i][0] * D[j][0] + D[i][1] * D[j][1] + D[i][2] * D[j][2] +
           D[i][3] * D[j][3];
  }
}

template <int BLK, int... L>
__device__ __forceinline__ void gram_block(float (&v)[16],
                                           const float (&D)[16][4],
                                           std::integer_sequence<int, L...>) {
  ((v[L] = gram_partial<16 * BLK + L>(D)), ...);
}

// Reduce-scatter of 16 per-lane partials: within each half-warp lane l ends
// with the half's sum of element l % 16, and one exchange across the halves
// completes the warp sum (held by lanes l and l + 16).
__device__ __forceinline__ float reduce_scatter16(float (&v)[16], int lane) {
#pragma unroll
  for (int o = 8; o >= 1; o >>= 1) {
    const bool hi = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      float send = hi ? v[i] : v[i + o];
      float keep = hi ? v[i + o] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 16);
}

// Gram block BLK (entries 16 BLK .. 16 BLK + 15 of the upper triangle) into
// both triangles of the slot-ordered matrix.
template <int BLK>
__device__ __forceinline__ void gram_store(const float (&D)[16][4],
                                           float (&A)[16][kAS], int lane) {
  float v[16];
  gram_block<BLK>(v, D, std::make_integer_sequence<int, 16>{});
  const float g = reduce_scatter16(v, lane);
  const int p = 16 * BLK + (lane & 15);
  if (lane < 16 && p < 136) {
    const int i = index_slot(pair_i(p)), j = index_slot(pair_j(p));
    A[i][j] = g;
    A[j][i] = g;
  }
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1)
    x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

// Quantise (storage paragraph of §4.1) and write one 832-byte record.
// V: lane-owned rows 4l..4l+3 of the fp32 basis; mu: lane-owned centroid
// entries; sm.post.Cf: fp32 coefficients [16][8].  vpage: one basis scale
// for the whole page (absolute maximum over every column), stored in all
// eight column slots; otherwise one per column.
// int4 codes and scale of basis column k (this lane's rows 4l..4l+3 in v);
// `apage` >= 0 is the page-wide absolute maximum (one scale per page),
// otherwise the column's own maximum is taken.
__device__ __forceinline__ void quantize_basis_column(int k, const float (&v)[4],
                                                      float apage,
                                                      BuildSmem &sm,
                                                      int lane) {
  float a = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])),
                  fmaxf(fabsf(v[2]), fabsf(v[3])));
  a = apage >= 0.f ? apage : warp_max(a);
  __half h = quant_scale(a, 7.f);
  float s = __half2float(h);
  if (lane == 0) sm.sv[k] = h;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    sm.post.v8[4 * lane + j][k] = (int8_t)quant_code(v[j], s, 7);
}

__device__ void write_record_tail(const float (&mu)[4], BuildSmem &sm,
                                  uint8_t *rec, int lane);

__device__ void write_record(const float (&V)[4][8], const float (&mu)[4],
                             BuildSmem &sm, uint8_t *rec, int lane,
                             bool vpage) {
  float apage = -1.f;
  if (vpage) {
    apage = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k)
#pragma unroll
      for (int j = 0; j < 4; ++j) apage = fmaxf(apage, fabsf(V[j][k]));
    apage = warp_max(apage);
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float v[4] = {V[0][k], V[1][k], V[2][k], V[3][k]};
    quantize_basis_column(k, v, apage, sm, lane);
  }
  write_record_tail(mu, sm, rec, lane);
}

// Everything of the record after the basis codes and scales (already in
// sm.post.v8 and sm.sv): the centroid, the coefficients and the packing.
__device__ void write_record_tail(const float (&mu)[4], BuildSmem &sm,
                                  uint8_t *rec, int lane) {
  // centroid: one scale, int8 codes
  {
    float a = fmaxf(fmaxf(fabsf(mu[0]), fabsf(mu[1])),
                    fmaxf(fabsf(mu[2]), fabsf(mu[3])));
    a = warp_max(a);
    __half h = quant_scale(a, 127.f);
    float s = __half2float(h);
    if (lane == 0) sm.smu = h;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      sm.post.m8[4 * lane + j] = (int8_t)quant_code(mu[j], s, 127);
  }
  __syncwarp();
  // coefficients: one scale per row (token), int8 codes
  if (lane < 16) {
    float a = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) a = fmaxf(a, fabsf(sm.post.Cf[lane][k]));
    __half h = quant_scale(a, 127.f);
    float s = __half2float(h);
    sm.sc[lane] = h;
#pragma unroll
    for (int k = 0; k < 8; ++k)
      sm.post.c8[lane][k] = (int8_t)quant_code(sm.post.Cf[lane][k], s, 127);
  }
  __syncwarp();
  // V4: lane t = 4n + c owns words (4n + c)*4 + w, w = 0..3
  {
    const int n = lane >> 2, c = lane & 3;
    uint32_t wv[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      uint32_t word = 0;
#pragma unroll
      for (int sp = 0; sp < 2; ++sp)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int d = 32 * w + 16 * sp + 8 * h + 2 * c + e;
            const uint32_t nib = (uint32_t)(sm.post.v8[d][n]) & 0xFu;
            word |= nib << (16 * e + 8 * sp + 4 * h);
          }
      wv[w] = word;
    }
    *reinterpret_cast<uint4 *>(rec + kOffV4 + 16 * lane) =
        make_uint4(wv[0], wv[1], wv[2], wv[3]);
  }
  // C8: lane t = 4*gi + c; int8 codes stored excess-128 (byte = code + 128,
  // i.e. the sign bit flipped)
  {
    const int gi = lane >> 2, c = lane & 3;
    uint32_t b0 = (uint8_t)sm.post.c8[gi][2 * c], b1 = (uint8_t)sm.post.c8[gi][2 * c + 1];
    uint32_t b2 = (uint8_t)sm.post.c8[gi + 8][2 * c];
    uint32_t b3 = (uint8_t)sm.post.c8[gi + 8][2 * c + 1];
    *reinterpret_cast<uint32_t *>(rec + kOffC8 + 4 * lane) =
        (b0 | (b1 << 8) | (b2 << 16) | (b3 << 24)) ^ 0x80808080u;
  }
  // MU8: lane l = 8c + s holds bytes d = 16s + 2c + {0, 1, 8, 9}
  {
    const int c = lane >> 3, s = lane & 7;
    const int d0 = 16 * s + 2 * c;
    uint32_t b0 = (uint8_t)sm.post.m8[d0], b1 = (uint8_t)sm.post.m8[d0 + 1];
    uint32_t b2 = (uint8_t)sm.post.m8[d0 + 8], b3 = (uint8_t)sm.post.m8[d0 + 9];
    *reinterpret_cast<uint32_t *>(rec + kOffMu8 + 4 * lane) =
        (b0 | (b1 << 8) | (b2 << 16) | (b3 << 24)) ^ 0x80808080u;
  }
  // scale block: 16 bytes per t = 0..3 at 768 + 16t holding sV[2t..2t+1],
  // sC[2t..2t+1], sC[8+2t..9+2t], then sMU (t = 0) or zero
  if (lane < 16) {
    const int t = lane >> 2, q = lane & 3;
    uint32_t lo = 0, hi = 0;
    if (q == 0) {
      lo = __half_as_ushort(sm.sv[2 * t]);
      hi = __half_as_ushort(sm.sv[2 * t + 1]);
    } else if (q == 1) {
      lo = __half_as_ushort(sm.sc[2 * t]);
      hi = __half_as_ushort(sm.sc[2 * t + 1]);
    } else if (q == 2) {
      lo = __half_as_ushort(sm.sc[8 + 2 * t]);
      hi = __half_as_ushort(sm.sc[9 + 2 * t]);
    } else if (t == 0) {
      lo = __half_as_ushort(sm.smu);
    }
    *reinterpret_cast<uint32_t *>(rec + kOffSV + 4 * lane) = lo | (hi << 16);
  }
  __syncwarp();
}

__device__ __forceinline__ void load_page_keys(const __nv_bfloat16 *page,
                                               float (&kx)[16][4], int lane) {
  const uint2 *src = reinterpret_cast<const uint2 *>(page);
#pragma unroll
  for (int t = 0; t < 16; ++t) {
    const uint2 raw = src[t * 32 + lane];
    kx[t][0] = bf16_lo(raw.x);
    kx[t][1] = bf16_hi(raw.x);
    kx[t][2] = bf16_lo(raw.y);
    kx[t][3] = bf16_hi(raw.y);
  }
}

__device__ __forceinline__ void center_keys(float (&kx)[16][4],
                                            const float (&mu)[4]) {
#pragma unroll
  for (int t = 0; t < 16; ++t)
#pragma unroll
    for (int j = 0; j < 4; ++j) kx[t][j] = __fsub_rn(kx[t][j], mu[j]);
}

// Rotation of the pair (p, q) that zeroes A[p][q]: t = tan(phi) is the
// smaller root of t^2 + 2 theta t - 1 = 0 with theta = (a_qq - a_pp) /
// (2 a_pq), c = 1 / sqrt(1 + t^2), s = t c.  Skipped (c = 1, s = 0) when
// |a_pq| <= 1e-7 sqrt(|a_pp a_qq|) or |a_pq| <= 1e-30.
__device__ __forceinline__ bool jacobi_rotation(float app, float aqq,
                                                float apq, float &c,
                                                float &s) {
  c = 1.f;
  s = 0.f;
  if (!(apq * apq > kJacobiRelTol * kJacobiRelTol * fabsf(app * aqq)) ||
      !(fabsf(apq) > 1e-30f))
    return false;
  const float theta = __fdividef(aqq - app, 2.f * apq);
  float t;
  if (fabsf(theta) > 1e15f) {
    t = __fdividef(0.5f, theta);
  } else {
    const float r = fmaf(theta, theta, 1.f);
    t = __fdividef(copysignf(1.f, theta), fabsf(theta) + r * rsqrtf(r));
  }
  c = rsqrtf(fmaf(t, t, 1.f));
  s = t * c;
  return true;
}

// A lane's fixed share of a Jacobi round: the rotation of pair pm = lane % 8
// (from the diagonal block (pm, pm)), the matrix blocks (grp + 4j, pm) for
// j = 0, 1 with grp = lane / 8, and rows 4 grp .. 4 grp + 3 of the vector
// columns 2 pm, 2 pm + 1 (held in registers).  Offsets are in floats within
// one buffer.
struct JacobiLane {
  int grp, pm;
  int o_d;           // A[2pm][2pm]
  int o_blk;         // A[2 grp][2 pm] (block j adds 8 kAS rows)
  int st[2][2][2];   // destination of block element (j, x, y)
};

__device__ __forceinline__ JacobiLane jacobi_lane(int lane) {
  JacobiLane L;
  L.grp = lane >> 3;
  L.pm = lane & 7;
  L.o_d = 2 * L.pm * kAS + 2 * L.pm;
  L.o_blk = 2 * L.grp * kAS + 2 * L.pm;
#pragma unroll
  for (int j = 0; j < 2; ++j)
#pragma unroll
    for (int x = 0; x < 2; ++x)
#pragma unroll
      for (int y = 0; y < 2; ++y)
        L.st[j][x][y] = slot_next(2 * (L.grp + 4 * j) + x) * kAS +
                        slot_next(2 * L.pm + y);
  return L;
}

// One round: reads matrix buffer A, writes An in the next round's slot
// order, and updates this lane's vector entries u0 (column 2 pm) and u1
// (column 2 pm + 1), rows 4 grp + t, moving them to the next round's slots.
// Returns whether this lane's pair rotated.
__device__ __forceinline__ int jacobi_round(const float *__restrict__ A,
                                            float *__restrict__ An,
                                            float (&u0)[4], float (&u1)[4],
                                            const JacobiLane &L) {
  float c, s;
  const int rot = jacobi_rotation(A[L.o_d], A[L.o_d + kAS + 1], A[L.o_d + 1],
                                  c, s);
  // the row pair of block j is pair grp + 4j, whose rotation lane grp + 4j
  // computed
  float cr[2], sr[2];
  cr[0] = __shfl_sync(0xffffffffu, c, L.grp);
  sr[0] = __shfl_sync(0xffffffffu, s, L.grp);
  cr[1] = __shfl_sync(0xffffffffu, c, L.grp + 4);
  sr[1] = __shfl_sync(0xffffffffu, s, L.grp + 4);
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const float2 x0 = *reinterpret_cast<const float2 *>(A + L.o_blk + 8 * j * kAS);
    const float2 x1 =
        *reinterpret_cast<const float2 *>(A + L.o_blk + 8 * j * kAS + kAS);
    // rows: J^T X
    const float r00 = cr[j] * x0.x - sr[j] * x1.x;
    const float r10 = sr[j] * x0.x + cr[j] * x1.x;
    const float r01 = cr[j] * x0.y - sr[j] * x1.y;
    const float r11 = sr[j] * x0.y + cr[j] * x1.y;
    // columns: (J^T X) J
    float y00 = c * r00 - s * r01;
    float y01 = s * r00 + c * r01;
    float y10 = c * r10 - s * r11;
    float y11 = s * r10 + c * r11;
    if (L.grp + 4 * j == L.pm && s != 0.f) {  // the pair's own 2x2 block
      y01 = 0.f;
      y10 = 0.f;
    }
    An[L.st[j][0][0]] = y00;
    An[L.st[j][0][1]] = y01;
    An[L.st[j][1][0]] = y10;
    An[L.st[j][1][1]] = y11;
  }
  // U <- U J, then the columns move with the slots: the next even slot 2m
  // takes pair m+1's even column (pair 0 keeps its own, pair 7 takes its
  // own odd one), the next odd slot 2m+1 takes pair m-1's odd column (pair
  // 0 takes pair 1's even one)
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const float a = u0[t], b = u1[t];
    const float r0 = c * a - s * b, r1 = s * a + c * b;
    const float dn = __shfl_down_sync(0xffffffffu, r0, 1);
    const float up = __shfl_up_sync(0xffffffffu, r1, 1);
    u0[t] = L.pm == 7 ? r1 : (L.pm == 0 ? r0 : dn);
    u1[t] = L.pm == 0 ? dn : up;
  }
  __syncwarp();
  return rot;
}

// Algorithm 1 up to the eigendecomposition, on one page-head held as
// kx[token][4 dims of this lane] (bf16 values widened to fp32): centres kx
// on the fp32 centroid mu (lane-owned entries), and leaves in sm the
// eigenvectors U (columns), the eigenvalues lam (descending, clipped at
// zero) and perm (column of U of the k-th eigenvalue).
__device__ void page_eigen(float (&kx)[16][4], float (&mu)[4], BuildSmem &sm,
                           int lane) {
  // Eq.(2): centroid (fp32, tokens summed in order, then /16) and deviations
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float acc = 0.f;
#pragma unroll
    for (int t = 0; t < 16; ++t) acc = __fadd_rn(acc, kx[t][j]);
    mu[j] = __fmul_rn(acc, 0.0625f);
  }
  center_keys(kx, mu);

  // Eq.(3): Gram matrix D D^T, 136 unique entries in 9 blocks of 16
  gram_store<0>(kx, sm.jac.Ab[0], lane);
  gram_store<1>(kx, sm.jac.Ab[0], lane);
  gram_store<2>(kx, sm.jac.Ab[0], lane);
  gram_store<3>(kx, sm.jac.Ab[0], lane);
  gram_store<4>(kx, sm.jac.Ab[0], lane);
  gram_store<5>(kx, sm.jac.Ab[0], lane);
  gram_store<6>(kx, sm.jac.Ab[0], lane);
  gram_store<7>(kx, sm.jac.Ab[0], lane);
  gram_store<8>(kx, sm.jac.Ab[0], lane);
  __syncwarp();

  // cyclic Jacobi in slot order (see slot_next): rounds alternate between
  // the two buffers, a sweep is 15 rounds, and the iteration stops after a
  // sweep in which no pair rotated (or after kMaxSweeps sweeps)
  const JacobiLane L = jacobi_lane(lane);
  float *A0 = &sm.jac.Ab[0][0][0], *A1 = &sm.jac.Ab[1][0][0];
  // eigenvector accumulator U, identity in slot order: this lane's entries
  // at rows 4 grp + t of columns 2 pm (u0) and 2 pm + 1 (u1)
  float u0[4], u1[4];
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    u0[t] = 4 * L.grp + t == 2 * L.pm ? 1.f : 0.f;
    u1[t] = 4 * L.grp + t == 2 * L.pm + 1 ? 1.f : 0.f;
  }
  int fin = 0, rotated = 0, left = 15, sweeps = 0;
  for (;;) {
    rotated |= jacobi_round(A0, A1, u0, u1, L);
    if (--left == 0) {
      if (!__any_sync(0xffffffffu, rotated) || ++sweeps >= kMaxSweeps) {
        fin = 1;
        break;
      }
      rotated = 0;
      left = 15;
    }
    rotated |= jacobi_round(A1, A0, u0, u1, L);
    if (--left == 0) {
      if (!__any_sync(0xffffffffu, rotated) || ++sweeps >= kMaxSweeps) {
        fin = 0;
        break;
      }
      rotated = 0;
      left = 15;
    }
  }

  // back to index order: eigenvalue and eigenvector of slot a belong to
  // index slot_index(a); the vectors' rows are in slot order as well
  if (lane < 16) sm.ev[slot_index(lane)] = sm.jac.Ab[fin][lane][lane];
  __syncwarp();  // post.U overlays the matrix buffers
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const int r = slot_index(4 * L.grp + t);
    sm.post.U[r][slot_index(2 * L.pm)] = u0[t];
    sm.post.U[r][slot_index(2 * L.pm + 1)] = u1[t];
  }
  __syncwarp();

  // eigenvalues descending (ties: lower index first), clipped at zero
  if (lane < 16) {
    const float li = sm.ev[lane];
    int rank = 0;
    for (int j = 0; j < 16; ++j) {
      const float lj = sm.ev[j];
      rank += (lj > li) || (lj == li && j < lane);
    }
    sm.perm[rank] = lane;
    sm.lam[rank] = fmaxf(li, 0.f);
  }
  __syncwarp();
}

// Sign rule and per-component factors of the first r components (lanes
// < r): U column perm[k] is signed so its largest-magnitude entry is
// positive (lowest index on exact ties); components with lam <= 1e-6 lam_1
// are zeroed.  cv = sign / sigma (basis), cc = sign * sigma (coefficients).
__device__ __forceinline__ void component_factors(const BuildSmem &sm, int r,
                                                  int lane, float *cv,
                                                  float *cc) {
  if (lane < r) {
    const int col = sm.perm[lane];
    float best = -1.f;
    int bi = 0;
    for (int i = 0; i < 16; ++i) {
      const float a = fabsf(sm.post.U[i][col]);
      if (a > best) {
        best = a;
        bi = i;
      }
    }
    const float sg = sm.post.U[bi][col] < 0.f ? -1.f : 1.f;
    const float lam = sm.lam[lane], lam1 = sm.lam[0];
    const bool keep = lam1 > 0.f && lam > 1e-6f * lam1;
    const float sig = sqrtf(lam);
    cv[lane] = keep ? sg / sig : 0.f;
    cc[lane] = keep ? sg * sig : 0.f;
  }
  __syncwarp();
}

// Algorithm 1 on the page-head at `page` (bf16 [16][128]; lane l handles
// dims 4l..4l+3).  Writes the record and returns tau (valid on every lane).
__device__ float summarize_page(const __nv_bfloat16 *page, BuildSmem &sm,
                                uint8_t *rec, int lane, bool vpage,
                                float *unq = nullptr) {
  float mu[4];
  float kx[16][4];
  load_page_keys(page, kx, lane);
  page_eigen(kx, mu, sm, lane);
  // the keys again (L2-resident), centred as before: not held in registers
  // through the eigensolve
  load_page_keys(page, kx, lane);
  center_keys(kx, mu);
  // sign rule and per-component factors
  component_factors(sm, kRank, lane, sm.cv, sm.cc);
  float tau = 0.f;
#pragma unroll
  for (int k = kRank; k < 16; ++k) tau += sm.lam[k];

  // V = D^T U_r Sigma_r^{-1}, one column at a time (this lane's rows),
  // quantised as soon as it is formed; with one scale per page the columns
  // are formed twice, the first time for the page maximum
  auto basis_column = [&](int k, float (&v)[4]) {
    const int col = sm.perm[k];
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float u = sm.post.U[i][col];
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[j] = fmaf(kx[i][j], u, acc[j]);
    }
    const float f = sm.cv[k];
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = acc[j] * f;
  };
  float apage = -1.f;
  if (vpage) {
    apage = 0.f;
#pragma unroll 1
    for (int k = 0; k < 8; ++k) {
      float v[4];
      basis_column(k, v);
      apage = fmaxf(apage, fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])),
                                 fmaxf(fabsf(v[2]), fabsf(v[3]))));
    }
    apage = warp_max(apage);
  }
#pragma unroll 1
  for (int k = 0; k < 8; ++k) {
    float v[4];
    basis_column(k, v);
    quantize_basis_column(k, v, apage, sm, lane);
    if (unq) {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        unq[16 + kDim + (4 * lane + j) * kRank + k] = v[j];
    }
  }
  // C = U_r Sigma_r (shared)
  {
    const int i = lane >> 1, k0 = (lane & 1) * 4;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const int k = k0 + kk;
      sm.post.Cf[i][k] = sm.post.U[i][sm.perm[k]] * sm.cc[k];
    }
  }
  __syncwarp();
  if (unq) {  // fp32 values before quantisation: lam, mu, (V above), C
    if (lane < 16) unq[lane] = sm.lam[lane];
    reinterpret_cast<float4 *>(unq + 16)[lane] =
        make_float4(mu[0], mu[1], mu[2], mu[3]);
    const int i = lane >> 1, k0 = (lane & 1) * 4;
    reinterpret_cast<float4 *>(unq + 16 + kDim + kDim * kRank)[lane] =
        make_float4(sm.post.Cf[i][k0], sm.post.Cf[i][k0 + 1], sm.post.Cf[i][k0 + 2],
                    sm.post.Cf[i][k0 + 3]);
  }
  write_record_tail(mu, sm, rec, lane);
  return tau;
}


// six CTAs (24 warps) per SM: the build is bound by the shared-memory data
// pipe and by latency, and 80 registers (a few bytes of spills outside the
// eigensolve) measured faster than 128 without spills
__global__ void __launch_bounds__(32 * kBuildWarps, 6)
    build_kernel(const __nv_bfloat16 *__restrict__ k_cache,
                 int64_t num_phys, int h_kv, const int32_t *__restrict__ pt,
                 int batch, int max_pages, const int32_t *__restrict__ seq_ids,
                 const int32_t *__restrict__ page_ids, int n_pairs,
                 uint8_t *__restrict__ summaries, float *__restrict__ tau_out,
                 float *__restrict__ unq_out, int flags, int32_t *status) {
  __shared__ BuildSmem smem[kBuildWarps];
  const bool vpage = (flags & LOCKS_BUILD_VSCALE_PER_PAGE) != 0;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  BuildSmem &sm = smem[wid];
  const long long total = (long long)n_pairs * h_kv;
  for (long long w = (long long)blockIdx.x * kBuildWarps + wid; w < total;
       w += (long long)gridDim.x * kBuildWarps) {
    const int pair = (int)(w / h_kv), h = (int)(w % h_kv);
    const int b = seq_ids[pair], pg = page_ids[pair];
    if (b < 0 || b >= batch || pg < 0 || pg >= max_pages) {
      if (lane == 0) set_status(status, LOCKS_DEV_BAD_PAIR);
      continue;
    }
    const int phys = pt[(size_t)b * max_pages + pg];
    if (phys < 0 || phys >= num_phys) {
      if (lane == 0) set_status(status, LOCKS_DEV_BAD_PAGE_ID);
      continue;
    }
    uint8_t *rec =
        summaries + (((size_t)b * h_kv + h) * max_pages + pg) * (size_t)kRec;
    const float tau = summarize_page(
        k_cache + ((size_t)phys * h_kv + h) * kPage * kDim, sm, rec, lane,
        vpage,
        unq_out ? unq_out + (size_t)w * LOCKS_UNQUANTISED_FLOATS : nullptr);
    if (tau_out && lane == 0) tau_out[w] = tau;
  }
}

__global__ void __launch_bounds__(32 * kBuildWarps)
    pack_kernel(const float *__restrict__ mu, const float *__restrict__ basis,
                const float *__restrict__ coeffs, int n,
                uint8_t *__restrict__ records, int flags) {
  __shared__ BuildSmem smem[kBuildWarps];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  BuildSmem &sm = smem[wid];
  for (long long w = (long long)blockIdx.x * kBuildWarps + wid; w < n;
       w += (long long)gridDim.x * kBuildWarps) {
    float m[4], V[4][8];
    const float4 mv = reinterpret_cast<const float4 *>(mu + w * kDim)[lane];
    m[0] = mv.x;
    m[1] = mv.y;
    m[2] = mv.z;
    m[3] = mv.w;
    const float4 *vb =
        reinterpret_cast<const float4 *>(basis + w * kDim * kRank) + lane * 8;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float4 a = vb[2 * j], c = vb[2 * j + 1];
      V[j][0] = a.x;
      V[j][1] = a.y;
      V[j][2] = a.z;
      V[j][3] = a.w;
      V[j][4] = c.x;
      V[j][5] = c.y;
      V[j][6] = c.z;
      V[j][7] = c.w;
    }
    const float4 cv =
        reinterpret_cast<const float4 *>(coeffs + w * kPage * kRank)[lane];
    const int i = lane >> 1, k0 = (lane & 1) * 4;
    sm.post.Cf[i][k0] = cv.x;
    sm.post.Cf[i][k0 + 1] = cv.y;
    sm.post.Cf[i][k0 + 2] = cv.z;
    sm.post.Cf[i][k0 + 3] = cv.w;
    __syncwarp();
    write_record(V, m, sm, records + w * (size_t)kRec, lane,
                 (flags & LOCKS_BUILD_VSCALE_PER_PAGE) != 0);
  }
}

// One CTA per sequence, one warp per KV head.
__global__ void append_kernel(const __nv_bfloat16 *__restrict__ k_new,
                              const __nv_bfloat16 *__restrict__ v_new,
                              __nv_bfloat16 *k_cache, __nv_bfloat16 *v_cache,
                              int64_t num_phys, int h_kv,
                              const int32_t *__restrict__ pt, int max_pages,
                              int32_t *seq_lens, uint8_t *summaries,
                              float *tau_out, int flags, int32_t *status) {
  extern __shared__ __align__(16) unsigned char append_smem[];
  BuildSmem *smem = reinterpret_cast<BuildSmem *>(append_smem);
  const int b = blockIdx.x;
  const int lane = threadIdx.x & 31, h = threadIdx.x >> 5;
  const int pos = seq_lens[b];
  __syncthreads();
  bool ok = pos >= 0 && pos < max_pages * kPage;
  int phys = -1;
  if (ok) {
    phys = pt[(size_t)b * max_pages + pos / kPage];
    if (phys < 0 || phys >= num_phys) {
      if (lane == 0 && h == 0) set_status(status, LOCKS_DEV_BAD_PAGE_ID);
      ok = false;
    }
  } else if (lane == 0 && h == 0) {
    set_status(status, LOCKS_DEV_BAD_SEQ_LEN);
  }
  if (ok) {
    const size_t page_off = ((size_t)phys * h_kv + h) * kPage * kDim;
    const size_t tok_off = page_off + (size_t)(pos % kPage) * kDim;
    const uint2 kv = reinterpret_cast<const uint2 *>(
        k_new + ((size_t)b * h_kv + h) * kDim)[lane];
    const uint2 vv = reinterpret_cast<const uint2 *>(
        v_new + ((size_t)b * h_kv + h) * kDim)[lane];
    reinterpret_cast<uint2 *>(k_cache + tok_off)[lane] = kv;
    reinterpret_cast<uint2 *>(v_cache + tok_off)[lane] = vv;
    if ((pos + 1) % kPage == 0) {
      // each lane re-reads exactly the bytes it wrote, so program order
      // makes the new token visible to this warp's build
      uint8_t *rec = summaries +
                     (((size_t)b * h_kv + h) * max_pages + pos / kPage) *
                         (size_t)kRec;
      const float tau =
          summarize_page(k_cache + page_off, smem[h], rec, lane,
                         (flags & LOCKS_BUILD_VSCALE_PER_PAGE) != 0);
      if (tau_out && lane == 0) tau_out[(size_t)b * h_kv + h] = tau;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && ok) seq_lens[b] = pos + 1;
}

// --------------------------------------------------------------------------
// rank / precision variants (notes §6 ablation): Algorithm 1 at rank R with
// a `vbits`-bit basis, written as a variant record (variant_layout.cuh,
// include/locks.h): codes are quantised per lane into shared memory, then
// each lane assembles whole words of the fragment-ordered record.
// --------------------------------------------------------------------------
struct VariantSmem {
  float cv[16], cc[16];
  float Cf[16][16];
  int8_t vq[kDim][16];  // basis codes [d][k]
  int8_t cq[16][16];    // coefficient codes [i][k]
};

template <int R>
__device__ float summarize_variant(const __nv_bfloat16 *page, BuildSmem &sm,
                                   VariantSmem &vs, uint8_t *rec, int vbits,
                                   int lane) {
  float mu[4];
  float kx[16][4];
  load_page_keys(page, kx, lane);
  page_eigen(kx, mu, sm, lane);
  load_page_keys(page, kx, lane);
  center_keys(kx, mu);
  component_factors(sm, R, lane, vs.cv, vs.cc);
  float tau = 0.f;
  for (int k = R; k < 16; ++k) tau += sm.lam[k];
  // V = D^T U_R Sigma_R^{-1} (lane rows), C = U_R Sigma_R (shared)
  float V[4][R];
#pragma unroll
  for (int k = 0; k < R; ++k) {
    const int col = sm.perm[k];
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float u = sm.post.U[i][col];
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[j] = fmaf(kx[i][j], u, acc[j]);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) V[j][k] = acc[j] * vs.cv[k];
  }
  for (int e = lane; e < 16 * R; e += 32) {
    const int i = e / R, k = e - i * R;
    vs.Cf[i][k] = sm.post.U[i][sm.perm[k]] * vs.cc[k];
  }
  const int off_c = var_off_c(R, vbits), off_mu = var_off_mu(R, vbits);
  const int off_s = var_off_s(R, vbits);
  // the scale block and the coefficient region start as zero scales and
  // zero codes (excess-128), so padding entries are defined
  for (int b = lane; b < 64; b += 32) rec[off_s + b] = 0;
  for (int b = lane; b < var_coeff_bytes(R); b += 32) rec[off_c + b] = 128;
  __syncwarp();
  const float qv = (float)((1 << (vbits - 1)) - 1);
  // basis: one scale per column; this lane's dims 4 lane .. 4 lane + 3
#pragma unroll
  for (int k = 0; k < R; ++k) {
    float a = fmaxf(fmaxf(fabsf(V[0][k]), fabsf(V[1][k])),
                    fmaxf(fabsf(V[2][k]), fabsf(V[3][k])));
    a = warp_max(a);
    const __half h = quant_scale(a, qv);
    if (lane == k)
      *reinterpret_cast<__half *>(rec + off_s + var_sv_off(k)) = h;
    const float sc = __half2float(h);
#pragma unroll
    for (int j = 0; j < 4; ++j)
      vs.vq[4 * lane + j][k] = (int8_t)quant_code(V[j][k], sc, (int)qv);
  }
  // centroid: one scale, int8 codes (excess-128)
  {
    float a = fmaxf(fmaxf(fabsf(mu[0]), fabsf(mu[1])),
                    fmaxf(fabsf(mu[2]), fabsf(mu[3])));
    a = warp_max(a);
    const __half h = quant_scale(a, 127.f);
    const float sc = __half2float(h);
    if (lane == 0)
      *reinterpret_cast<__half *>(rec + var_off_smu(R, vbits)) = h;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      rec[off_mu + var_mu_off(4 * lane + j)] =
          (uint8_t)(quant_code(mu[j], sc, 127) + 128);
  }
  // coefficients: one scale per row (token), int8 codes
  if (lane < 16) {
    float a = 0.f;
    for (int k = 0; k < R; ++k) a = fmaxf(a, fabsf(vs.Cf[lane][k]));
    const __half h = quant_scale(a, 127.f);
    const float sc = __half2float(h);
    *reinterpret_cast<__half *>(rec + off_s + var_sc_off(lane)) = h;
    for (int k = 0; k < R; ++k) {
      const int c = quant_code(vs.Cf[lane][k], sc, 127);
      rec[off_c + var_c_off(R, lane, k)] = (uint8_t)(c + 128);
    }
  }
  __syncwarp();
  // basis words: word wi of slot (k, t) = (wi / vbits) holds the codes of
  // the dims var_v_bit places there
  const uint32_t cmask = (1u << vbits) - 1u;
  const int n_words = 4 * R * vbits;
  for (int wi = lane; wi < n_words; wi += 32) {
    const int slot = wi / vbits, w = wi - slot * vbits;
    const int k = slot >> 2, t = slot & 3;
    const int spw = 8 / vbits;  // k-steps per word
    uint32_t word = 0;
    for (int s = w * spw; s < (w + 1) * spw; ++s)
      for (int e = 0; e < 2; ++e)
        for (int h = 0; h < 2; ++h) {
          const int d = 16 * s + 2 * t + e + 8 * h;
          const int c = vs.vq[d][k];
          const uint32_t u = vbits == 8 ? (uint32_t)(c + 128)
                                        : (uint32_t)c & cmask;
          word |= u << (var_v_bit(vbits, d, k) - 32 * wi);
        }
    reinterpret_cast<uint32_t *>(rec)[wi] = word;
  }
  __syncwarp();
  return tau;
}

template <int R>
__global__ void __launch_bounds__(32 * kBuildWarps, 4)
    build_variant_kernel(const __nv_bfloat16 *__restrict__ k_cache,
                         int64_t num_phys, int h_kv,
                         const int32_t *__restrict__ pt, int batch,
                         int max_pages, const int32_t *__restrict__ seq_ids,
                         const int32_t *__restrict__ page_ids, int n_pairs,
                         int vbits, uint8_t *__restrict__ records,
                         float *__restrict__ tau_out, int32_t *status) {
  __shared__ BuildSmem smem[kBuildWarps];
  __shared__ VariantSmem vsm[kBuildWarps];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const size_t stride = (size_t)var_stride(R, vbits);
  const long long total = (long long)n_pairs * h_kv;
  for (long long w = (long long)blockIdx.x * kBuildWarps + wid; w < total;
       w += (long long)gridDim.x * kBuildWarps) {
    const int pair = (int)(w / h_kv), h = (int)(w % h_kv);
    const int b = seq_ids[pair], pg = page_ids[pair];
    if (b < 0 || b >= batch || pg < 0 || pg >= max_pages) {
      if (lane == 0) set_status(status, LOCKS_DEV_BAD_PAIR);
      continue;
    }
    const int phys = pt[(size_t)b * max_pages + pg];
    if (phys < 0 || phys >= num_phys) {
      if (lane == 0) set_status(status, LOCKS_DEV_BAD_PAGE_ID);
      continue;
    }
    uint8_t *rec =
        records + (((size_t)b * h_kv + h) * max_pages + pg) * stride;
    const float tau = summarize_variant<R>(
        k_cache + ((size_t)phys * h_kv + h) * kPage * kDim, smem[wid],
        vsm[wid], rec, vbits, lane);
    if (tau_out && lane == 0) tau_out[w] = tau;
  }
}

// --------------------------------------------------------------------------
// launchers
// --------------------------------------------------------------------------
static int grid_for(long long warps, int warps_per_cta) {
  long long g = (warps + warps_per_cta - 1) / warps_per_cta;
  if (g > 65535LL * 32) g = 65535LL * 32;
  return (int)(g < 1 ? 1 : g);
}

cudaError_t launch_build(const void *k_cache, int64_t num_phys, int h_kv,
                         const int32_t *pt, int batch, int max_pages,
                         const int32_t *seq_ids, const int32_t *page_ids,
                         int n_pairs, void *summaries, float *tau_out,
                         float *unq_out, int flags, int32_t *status,
                         cudaStream_t stream) {
  const long long warps = (long long)n_pairs * h_kv;
  if (warps == 0) return cudaSuccess;
  build_kernel<<<grid_for(warps, kBuildWarps), 32 * kBuildWarps, 0, stream>>>(
      static_cast<const __nv_bfloat16 *>(k_cache), num_phys, h_kv, pt, batch,
      max_pages, seq_ids, page_ids, n_pairs,
      static_cast<uint8_t *>(summaries), tau_out, unq_out, flags, status);
  return launched();
}

cudaError_t launch_build_variant(const void *k_cache, int64_t num_phys,
                                 int h_kv, const int32_t *pt, int batch,
                                 int max_pages, const int32_t *seq_ids,
                                 const int32_t *page_ids, int n_pairs,
                                 int rank, int vbits, void *records,
                                 float *tau_out, int32_t *status,
                                 cudaStream_t stream) {
  const long long warps = (long long)n_pairs * h_kv;
  if (warps == 0) return cudaSuccess;
  const int grid = grid_for(warps, kBuildWarps);
  auto *kc = static_cast<const __nv_bfloat16 *>(k_cache);
  auto *rec = static_cast<uint8_t *>(records);
#define LOCKS_BUILD_VARIANT(R)                                              \
  build_variant_kernel<R><<<grid, 32 * kBuildWarps, 0, stream>>>(           \
      kc, num_phys, h_kv, pt, batch, max_pages, seq_ids, page_ids, n_pairs, \
      vbits, rec, tau_out, status)
  switch (rank) {
    case 4: LOCKS_BUILD_VARIANT(4); break;
    case 8: LOCKS_BUILD_VARIANT(8); break;
    case 12: LOCKS_BUILD_VARIANT(12); break;
    case 15: LOCKS_BUILD_VARIANT(15); break;
    default: return cudaErrorInvalidValue;
  }
#undef LOCKS_BUILD_VARIANT
  return launched();
}

cudaError_t launch_pack(const float *mu, const float *basis,
                        const float *coeffs, int n, void *records, int flags,
                        cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  pack_kernel<<<grid_for(n, kBuildWarps), 32 * kBuildWarps, 0, stream>>>(
      mu, basis, coeffs, n, static_cast<uint8_t *>(records), flags);
  return launched();
}

cudaError_t launch_append(const void *k_new, const void *v_new, void *k_cache,
                          void *v_cache, int64_t num_phys, int h_kv,
                          const int32_t *pt, int batch, int max_pages,
                          int32_t *seq_lens, void *summaries, float *tau_out,
                          int flags, int32_t *status, cudaStream_t stream) {
  if (batch == 0) return cudaSuccess;
  const size_t smem = sizeof(BuildSmem) * (size_t)h_kv;
  static DeviceFlags attr_set;
  cudaError_t e = once_per_device(attr_set, [] {
    return cudaFuncSetAttribute(append_kernel,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)(sizeof(BuildSmem) * 32));
  });
  if (e != cudaSuccess) return e;
  append_kernel<<<batch, 32 * h_kv, smem, stream>>>(
      static_cast<const __nv_bfloat16 *>(k_new),
      static_cast<const __nv_bfloat16 *>(v_new),
      static_cast<__nv_bfloat16 *>(k_cache),
      static_cast<__nv_bfloat16 *>(v_cache), num_phys, h_kv, pt, max_pages,
      seq_lens, static_cast<uint8_t *>(summaries), tau_out, flags, status);
  return launched();
}

}  // namespace locks
