// Device helpers shared by the decode FFN kernels (decode_ffn.cu, the
// two-kernel path; decode_fused.cu, the one-pass fused kernel): mbarrier and
// bulk-copy wrappers with bounded waits, weight decoding (fp32, bf16, OCP
// e4m3) and activation loads.  Internal to libft.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "ft_internal.h"

namespace ft {
namespace dec {

constexpr unsigned long long kWaitLimitNs = 1000000000ull;

template <int WT> struct W;
template <> struct W<FT_W_F32> { static constexpr int kEPC = 4; static constexpr int kBytes = 4; };
template <> struct W<FT_W_BF16> { static constexpr int kEPC = 8; static constexpr int kBytes = 2; };
template <> struct W<FT_W_FP8E4M3_B128> { static constexpr int kEPC = 16; static constexpr int kBytes = 1; };

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_init_fence() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_n(uint64_t* bar, uint32_t n) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(n) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Bounded wait for phase `parity` of `bar`; false (and FT_ERR_TIMEOUT in
// *status) if it did not complete within the limit.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int32_t* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (;;) {
    for (int i = 0; i < 256; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > kWaitLimitNs) {
      if (status) atomicCAS(status, 0, (int)FT_ERR_TIMEOUT);
      return false;
    }
  }
}
// Bulk asynchronous copy global -> shared, completion counted on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_addr(dst)),
               "l"(src), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}
// Copy-engine mode: wait (bounded) until the library's host thread has set
// the ready flag of this layer's event, which it does on the copy stream after
// the event's blob copies.  Called by one thread before any weight read.
__device__ __forceinline__ void wait_ready_flag(const FfnArgs& a) {
  if (!a.ready_flags) return;
  const int ev = __ldg(&a.hdr[PH_EVENT]);
  const int32_t* f = a.ready_flags + (ev % kRing);
  const unsigned long long t0 = global_ns();
  for (;;) {
    int v;
    asm volatile("ld.acquire.sys.global.b32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
    if (v == ev) return;
    if (global_ns() - t0 > kWaitLimitNs) {
      if (a.status) atomicCAS(a.status, 0, (int)FT_ERR_TIMEOUT);
      return;
    }
  }
}
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait_primary() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------- decode helpers
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

template <int WT>
__device__ __forceinline__ void decode_chunk(const uint4& c, float* w);
template <>
__device__ __forceinline__ void decode_chunk<FT_W_F32>(const uint4& c, float* w) {
  w[0] = __uint_as_float(c.x); w[1] = __uint_as_float(c.y);
  w[2] = __uint_as_float(c.z); w[3] = __uint_as_float(c.w);
}
template <>
__device__ __forceinline__ void decode_chunk<FT_W_BF16>(const uint4& c, float* w) {
  w[0] = bf16_lo(c.x); w[1] = bf16_hi(c.x); w[2] = bf16_lo(c.y); w[3] = bf16_hi(c.y);
  w[4] = bf16_lo(c.z); w[5] = bf16_hi(c.z); w[6] = bf16_lo(c.w); w[7] = bf16_hi(c.w);
}
__device__ __forceinline__ void fp8x4(uint32_t v, float* w) {
  const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(v & 0xffffu), __NV_E4M3);
  const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(v >> 16), __NV_E4M3);
  const float2 a = __half22float2(__half2(lo));
  const float2 b = __half22float2(__half2(hi));
  w[0] = a.x; w[1] = a.y; w[2] = b.x; w[3] = b.y;
}
template <>
__device__ __forceinline__ void decode_chunk<FT_W_FP8E4M3_B128>(const uint4& c, float* w) {
  fp8x4(c.x, w); fp8x4(c.y, w + 4); fp8x4(c.z, w + 8); fp8x4(c.w, w + 12);
}

// N activations starting at element i of a row (f32 or bf16) -> floats.
template <bool kActF32, int N>
__device__ __forceinline__ void load_act(const uint8_t* row, int i, float* x) {
  if (kActF32) {
    const float4* p = reinterpret_cast<const float4*>(row) + i / 4;
#pragma unroll
    for (int q = 0; q < N / 4; ++q) {
      const float4 v = p[q];
      x[4 * q] = v.x; x[4 * q + 1] = v.y; x[4 * q + 2] = v.z; x[4 * q + 3] = v.w;
    }
  } else {
    const uint4* p = reinterpret_cast<const uint4*>(row) + i / 8;
#pragma unroll
    for (int q = 0; q < N / 8; ++q) {
      const uint4 v = p[q];
      x[8 * q] = bf16_lo(v.x); x[8 * q + 1] = bf16_hi(v.x); x[8 * q + 2] = bf16_lo(v.y);
      x[8 * q + 3] = bf16_hi(v.y); x[8 * q + 4] = bf16_lo(v.z); x[8 * q + 5] = bf16_hi(v.z);
      x[8 * q + 6] = bf16_lo(v.w); x[8 * q + 7] = bf16_hi(v.w);
    }
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float scale_at(const uint8_t* blob, long long scale_off, int idx) {
  const uint16_t s = __ldg(reinterpret_cast<const uint16_t*>(blob + scale_off) + idx);
  return __uint_as_float((uint32_t)s << 16);
}

__host__ __device__ __forceinline__ int align_up(int v, int a) { return (v + a - 1) / a * a; }



}  // namespace dec
}  // namespace ft
