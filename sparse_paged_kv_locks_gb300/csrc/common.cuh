// Shared device helpers of the LOCKS kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "locks.h"

namespace locks {

constexpr int kPage = LOCKS_PAGE_TOKENS;  // B
constexpr int kDim = LOCKS_HEAD_DIM;      // d
constexpr int kRank = LOCKS_RANK;         // r
constexpr int kRec = LOCKS_RECORD_BYTES;  // record stride
constexpr int kOffV4 = 0, kOffC8 = 512, kOffMu8 = 640;
constexpr int kOffSV = 768;   // 64-byte scale block (see include/locks.h)
constexpr int kOffSMu = 780;
constexpr int kMaxGroup = 16;
constexpr size_t kWsHeader = 256;  // status word + reserved

__device__ __forceinline__ void set_status(int32_t *status, int bits) {
  if (status) atomicOr(status, bits);
}

// ---------------------------------------------------------------------------
// programmatic dependent launch: a kernel of the decode step lets the next
// one launch while it runs (pdl_trigger), and the next one waits for the
// previous grid to finish, with its memory visible, before it touches that
// grid's outputs or any buffer the previous grid reads (pdl_wait).  A kernel
// launched without a programmatic predecessor returns from pdl_wait at once.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
}
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// Launch with programmatic stream serialisation allowed (host side).
// kernels this process launched through the library (api.cu; read by
// locks_kernel_launches)
extern std::atomic<long long> g_kernel_launches;
inline void note_launches(long long n = 1) {
  g_kernel_launches.fetch_add(n, std::memory_order_relaxed);
}
// after a <<<...>>> launch: its error, counting it when it succeeded
inline cudaError_t launched() {
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) note_launches();
  return e;
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block,
                              size_t smem, cudaStream_t stream,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e =
      cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
  if (e == cudaSuccess) note_launches();
  return e;
}

// launch_pdl with thread-block clusters of `cluster` CTAs along x
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl_cluster(void (*kern)(KArgs...), dim3 grid,
                                      dim3 block, size_t smem,
                                      cudaStream_t stream, int cluster,
                                      Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const cudaError_t e =
      cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
  if (e == cudaSuccess) note_launches();
  return e;
}

// ---------------------------------------------------------------------------
// quantiser (storage paragraph of §4.1): symmetric, fp16 scale
// ---------------------------------------------------------------------------
__device__ __forceinline__ __half quant_scale(float absmax, float qmax) {
  float s = __fdiv_rn(absmax, qmax);
  __half h = __float2half_rn(s);
  if (__hisinf(h)) h = __ushort_as_half((unsigned short)0x7BFF);  // 65504
  return h;
}

__device__ __forceinline__ int quant_code(float x, float s, int qmax) {
  if (s == 0.f) return 0;
  int c = __float2int_rn(__fdiv_rn(x, s));
  return max(-qmax, min(qmax, c));
}

// ---------------------------------------------------------------------------
// tensor-core and copy primitives (inline PTX)
// ---------------------------------------------------------------------------
// D += A * B, m16n8k16, fp16 inputs, fp32 accumulators
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4],
                                        uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D += A * B, m16n8k16, bf16 inputs, fp32 accumulators
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4],
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile(
      "ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x2(uint32_t (&r)[2], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];\n"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4],
                                                  uint32_t addr) {
  asm volatile(
      "ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "r"(addr));
}

// 16-byte asynchronous global->shared copy (L2 only)
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst),
               "l"(src));
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::);
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

// mbarrier + 1-D bulk copy (TMA engine, no tensor map)
__device__ __forceinline__ void mbar_init(uint64_t *bar, int count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(
                   smem_u32(bar)),
               "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::);
}
__device__ __forceinline__ void mbar_arrive_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile(
      "mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::
          "r"(smem_u32(bar)),
      "r"(bytes)
      : "memory");
}
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src,
                                         uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1], %2, [%3];\n" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t phase) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(phase)
      : "memory");
  return ok != 0;
}
// Bounded wait: false when the barrier did not complete in `limit` tries.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t phase,
                                          uint32_t limit = (1u << 22)) {
  for (uint32_t i = 0; i < limit; ++i)
    if (mbar_try_wait(bar, phase)) return true;
  return false;
}

// ---------------------------------------------------------------------------
// thread-block clusters: rank, size, distributed shared memory, barrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;\n" : "=r"(r));
  return r;
}
// shared::cluster address of this CTA's shared-memory address `a` in the
// CTA of rank `rank`
__device__ __forceinline__ uint32_t mapa_shared(uint32_t a, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n"
               : "=r"(r)
               : "r"(a), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_u32(uint32_t a, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;\n" ::"r"(a), "r"(v)
               : "memory");
}
__device__ __forceinline__ void st_cluster_v4(uint32_t a, uint4 v) {
  asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};\n" ::"r"(a),
               "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void st_cluster_f32(uint32_t a, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;\n" ::"r"(a), "f"(v)
               : "memory");
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t a) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];\n" : "=f"(v) : "r"(a)
               : "memory");
  return v;
}
__device__ __forceinline__ float4 ld_cluster_v4f(uint32_t a) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];\n"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(a)
               : "memory");
  return v;
}
// every thread of every CTA of the cluster; orders the shared-memory
// (local and distributed) accesses before it against those after it
__device__ __forceinline__ void cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n"
      "barrier.cluster.wait.acquire.aligned;\n" ::
          : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];\n" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds16(uint32_t a) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];\n" : "=h"(v) : "r"(a));
  return v;
}

// D = A * B + C with separate C registers, m16n8k16, bf16 inputs
__device__ __forceinline__ void mma_bf16_c(float (&d)[4],
                                           const uint32_t (&a)[4],
                                           uint32_t b0, uint32_t b1,
                                           float c0, float c1, float c2,
                                           float c3) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%11,%12,%13};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1),
        "f"(c0), "f"(c1), "f"(c2), "f"(c3));
}

// D = A * B (zero accumulator), m16n8k8, fp16 inputs
__device__ __forceinline__ void mma1688_f16_z(float (&d)[4], uint32_t a0,
                                              uint32_t a1, uint32_t b0) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5}, {%6}, {%7,%7,%7,%7};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(b0), "f"(0.f));
}

// 8x8 transpose of 16-bit elements across the warp (thread t holds row t/4,
// elements 2(t%4) and 2(t%4)+1, before and after)
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n"
               : "=r"(y)
               : "r"(x));
  return y;
}

__device__ __forceinline__ uint4 ld_shared_v4(const void *p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_u32(p)));
  return v;
}
__device__ __forceinline__ uint32_t ld_shared_u32(const void *p) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];\n" : "=r"(v) : "r"(smem_u32(p)));
  return v;
}

// ---------------------------------------------------------------------------
// code -> fp16 conversions (exact small integers)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t lop3_and_xor(uint32_t x, uint32_t m,
                                                 uint32_t c) {
  uint32_t r;
  // r = (x & m) ^ c
  asm("lop3.b32 %0, %1, %2, %3, 0x6a;\n" : "=r"(r) : "r"(x), "r"(m), "r"(c));
  return r;
}

__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) {
  return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) {
  return *reinterpret_cast<__half2 *>(&u);
}

// Two int4 codes at bits [0,4) and [16,20) of x -> half2 (exact).
// (x & 0x000F000F) ^ 0x64086408 = 1024 + (code + 8) per half; minus 1032.
__device__ __forceinline__ uint32_t nib_lo_to_h2(uint32_t x) {
  uint32_t v = lop3_and_xor(x, 0x000F000Fu, 0x64086408u);
  return h2_as_u32(__hsub2(u32_as_h2(v), __half2half2(__ushort_as_half(
                                             (unsigned short)0x6408))));
}
// Two int4 codes at bits [4,8) and [20,24) of x -> half2 (exact).
// (x & 0x00F000F0) ^ 0x64806480 = 1152 + 16*code; times 1/16 minus 72.
__device__ __forceinline__ uint32_t nib_hi_to_h2(uint32_t x) {
  uint32_t v = lop3_and_xor(x, 0x00F000F0u, 0x64806480u);
  return h2_as_u32(__hfma2(u32_as_h2(v),
                           __half2half2(__ushort_as_half((unsigned short)0x2C00)),
                           __half2half2(__ushort_as_half((unsigned short)0xD480))));
}
// Two int8 codes in the low 16 bits of x -> half2 (exact):
// prmt places the bytes under 0x64 exponent bytes after flipping the sign
// bit (1152 + code), then subtract 1152.
__device__ __forceinline__ uint32_t i8x2_to_h2(uint32_t x) {
  uint32_t f = x ^ 0x00008080u;
  uint32_t v;
  asm("prmt.b32 %0, %1, %2, 0x7170;\n" : "=r"(v) : "r"(f), "r"(0x64646464u));
  return h2_as_u32(__hsub2(u32_as_h2(v), __half2half2(__ushort_as_half(
                                             (unsigned short)0x6480))));
}

__device__ __forceinline__ float bf16_lo(uint32_t u) {
  return __uint_as_float(u << 16);
}
__device__ __forceinline__ float bf16_hi(uint32_t u) {
  return __uint_as_float(u & 0xFFFF0000u);
}

// Hardware base-2 exponential and logarithm (PTX approximate forms, relative
// error ~2^-22), used for the 16-token log-sum-exp of a page.
__device__ __forceinline__ float ex2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2_fast(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace locks
