// Device helpers shared by the summary scoring kernels (the shipped
// record's and the rank / precision variants'): code-to-fp16 operand
// conversions, mma.sync wrappers, the per-quad log-sum-exp forms, the
// L2 policy of the score stores and the per-warp tile cursor.
#pragma once
#include "common.cuh"

namespace locks {

// log2(e) / sqrt(128): logits are carried in base-2 units
constexpr float kLog2eRsqrtD = 0.12751743074602467f;
constexpr float kLn2 = 0.69314718055994531f;

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  return h2_as_u32(__floats2half2_rn(lo, hi));
}

// fp16x2 of (p0 - h.x, p1 - h.y) for h = fp16x2(p0, p1): the low halves of a
// two-term fp16 split (both differences are exact in fp32; mixed-precision
// fma takes h's halves without converting them first)
__device__ __forceinline__ uint32_t split_lo(uint32_t h, float p0, float p1) {
  float l0, l1;
  asm("{\n .reg .b16 a, b, m1;\n mov.b32 {a, b}, %2;\n"
      " mov.b16 m1, 0xBC00;\n"
      " fma.rn.f32.f16 %0, a, m1, %3;\n"
      " fma.rn.f32.f16 %1, b, m1, %4;\n}\n"
      : "=f"(l0), "=f"(l1)
      : "r"(h), "f"(p0), "f"(p1));
  return pack_h2(l0, l1);
}

// Two int4 codes at bits [0,4) and [16,20) -> bf16x2 holding 136 + code
// (exact); the constant 136 is cancelled through the accumulator's initial
// value, so no subtraction is spent per element.
__device__ __forceinline__ uint32_t nib_bf16_off(uint32_t x) {
  return lop3_and_xor(x, 0x000F000Fu, 0x43084308u);
}

// Four int8 codes stored excess-128 (byte = code + 128) -> two fp16x2
// holding 1024 + byte = 1152 + code (exact); the constant is cancelled
// through the accumulator's initial value.
__device__ __forceinline__ void i8x4_to_h2_off(uint32_t x, uint32_t &lo,
                                               uint32_t &hi) {
  asm("prmt.b32 %0, %1, %2, 0x7170;\n" : "=r"(lo) : "r"(x), "r"(0x64646464u));
  asm("prmt.b32 %0, %1, %2, 0x7372;\n" : "=r"(hi) : "r"(x), "r"(0x64646464u));
}

// Four int8 codes -> two fp16x2 holding the codes exactly.
__device__ __forceinline__ void i8x4_to_h2(uint32_t x, uint32_t &lo,
                                           uint32_t &hi) {
  uint32_t a, b;
  i8x4_to_h2_off(x, a, b);
  const __half2 k = __half2half2(__ushort_as_half((unsigned short)0x6480));
  lo = h2_as_u32(__hsub2(u32_as_h2(a), k));
  hi = h2_as_u32(__hsub2(u32_as_h2(b), k));
}

// Two int4 codes at bits [0,4) and [16,20) -> fp16x2 holding 1032 + code;
// at bits [4,8) and [20,24) -> fp16x2 holding 1152 + 16 code (exact).  An
// fp16 half has room for two code positions, a bf16 half for one, so the
// fp16 form needs one shift per four code pairs instead of three.
__device__ __forceinline__ uint32_t nib_f16_lo(uint32_t x) {
  return lop3_and_xor(x, 0x000F000Fu, 0x64086408u);
}
__device__ __forceinline__ uint32_t nib_f16_hi(uint32_t x) {
  return lop3_and_xor(x, 0x00F000F0u, 0x64806480u);
}

// D = A * B + C, m16n8k16 fp16
__device__ __forceinline__ void mma_f16_c(float (&d)[4],
                                          const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1, float c0, float c1,
                                          float c2, float c3) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%11,%12,%13};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1),
        "f"(c0), "f"(c1), "f"(c2), "f"(c3));
}

// D = A * B (zero accumulator), m16n8k16 fp16
__device__ __forceinline__ void mma_f16_z(float (&d)[4],
                                          const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1),
        "f"(0.f));
}

// log2-sum-exp2 of 16 logits spread 4 per lane over a quad, with the
// maximum subtracted first (always finite)
__device__ __forceinline__ float lse2_quad(float a, float b, float c,
                                           float d) {
  float m = fmaxf(fmaxf(a, b), fmaxf(c, d));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
  float e = (ex2_fast(a - m) + ex2_fast(b - m)) +
            (ex2_fast(c - m) + ex2_fast(d - m));
  e += __shfl_xor_sync(0xffffffffu, e, 1);
  e += __shfl_xor_sync(0xffffffffu, e, 2);
  return m + lg2_fast(e);
}

// Same value without the max pass: sums 2^x directly and falls back to the
// max-subtracted form for the whole warp when any quad's sum overflows or
// underflows (logits beyond about +-126 in base-2 units).
__device__ __forceinline__ float lse2_quad_fast(float a, float b, float c,
                                                float d) {
  float e = (ex2_fast(a) + ex2_fast(b)) + (ex2_fast(c) + ex2_fast(d));
  e += __shfl_xor_sync(0xffffffffu, e, 1);
  e += __shfl_xor_sync(0xffffffffu, e, 2);
  const bool bad = !(e > 0.f) || !(e < INFINITY);
  if (__any_sync(0xffffffffu, bad)) return lse2_quad(a, b, c, d);
  return lg2_fast(e);
}

// Same value without the max pass and without the check: the caller folds
// `bits(e) - bits(FLT_MIN)` into `bad` (unsigned max) and recomputes the
// tile with lse2_quad when any quad sum was zero, subnormal, inf or NaN.
__device__ __forceinline__ float lse2_quad_raw(float a, float b, float c,
                                               float d, uint32_t &bad) {
  float e = (ex2_fast(a) + ex2_fast(b)) + (ex2_fast(c) + ex2_fast(d));
  e += __shfl_xor_sync(0xffffffffu, e, 1);
  e += __shfl_xor_sync(0xffffffffu, e, 2);
  bad = max(bad, __float_as_uint(e) - 0x00800000u);
  return lg2_fast(e);
}
constexpr uint32_t kLseBad = 0x7F000000u;  // bad >= this: recompute

__device__ __forceinline__ float lse2_quad_sel(float a, float b, float c,
                                               float d, bool safe,
                                               uint32_t &bad) {
  return safe ? lse2_quad(a, b, c, d) : lse2_quad_raw(a, b, c, d, bad);
}

// L2 policy for the scores: kept in L2 ahead of the summary stream, so the
// selection kernel that follows reads them from L2
__device__ __forceinline__ uint64_t l2_keep_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;\n"
               : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void st_keep(float *p, float v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;\n" ::"l"(p),
               "f"(v), "l"(pol)
               : "memory");
}

// position of a warp in its contiguous range of tiles
struct Cursor {
  int b, h, j;
};

__device__ __forceinline__ void advance_cursor(Cursor &c, const int *tph,
                                               int batch, int h_kv) {
  if (++c.j == tph[c.b]) {
    c.j = 0;
    if (++c.h == h_kv) {
      c.h = 0;
      do {
        ++c.b;
      } while (c.b < batch && tph[c.b] == 0);
    }
  }
}

}  // namespace locks
