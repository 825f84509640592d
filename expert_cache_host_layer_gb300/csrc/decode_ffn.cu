// Decode-path expert FFN (T <= 8 tokens): two HBM-bound GEMV kernels that read
// the expert weights straight from their cache slots.
//
//   gate_up:  h[row][r] = silu(Wg[r] . x_t) * (Wu[r] . x_t)   for every row
//             (t, j) of every unique expert u and every r < I
//   down:     y[t][c]  = sum_u sum_(rows (t,j) of u) w_tj * (Wd[c] . h[row])   (fp32 y)
//
// One warp per task: a (unique expert, intermediate row) pair for gate_up, an
// output column c for down.  Each lane streams 16-byte chunks of the weight
// rows with all its loads issued before the arithmetic, so a CTA keeps many
// KB in flight; x is staged in shared memory, h (fp32, tiny) comes from L2.
// The combine is deterministic: the down task sums its experts in ascending
// expert order with no atomics.  fp8 weights are decoded in registers and
// scaled once per 16-element chunk (a chunk never crosses a 128-wide block).
//
// The SwiGLU expert and the gate-weighted combine follow the routed experts
// of the Qwen3-MoE / DeepSeek MoE layers the pages serve ("FreeToken vs vLLM
// on one RTX 3090", "Why the performance differs"; "FreeToken: Efficient
// Edge-Native MoE Serving ...", design paragraph: the FFN reads experts from
// the GPU expert cache).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "ft_internal.h"

namespace ft {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxRows = kDecodeMaxTokens;  // rows of one expert in a decode batch

template <int WT> struct W;
template <> struct W<FT_W_F32> { static constexpr int kEPC = 4; static constexpr int kBytes = 4; };
template <> struct W<FT_W_BF16> { static constexpr int kEPC = 8; static constexpr int kBytes = 2; };
template <> struct W<FT_W_FP8E4M3_B128> { static constexpr int kEPC = 16; static constexpr int kBytes = 1; };

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// Decode one 16-byte chunk of weights into kEPC floats.
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

__device__ __forceinline__ uint4 ldg16(const void* p) { return __ldg(static_cast<const uint4*>(p)); }

// kEPC activations starting at element i of a row (f32 or bf16) -> floats.
template <bool kActF32>
__device__ __forceinline__ void load_act(const void* row, int i, float* x, int n) {
  if (kActF32) {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(row) + i);
    for (int q = 0; q < n / 4; ++q) {
      const float4 v = p[q];
      x[4 * q] = v.x; x[4 * q + 1] = v.y; x[4 * q + 2] = v.z; x[4 * q + 3] = v.w;
    }
  } else {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(row) + i);
    for (int q = 0; q < n / 8; ++q) {
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

// ---------------------------------------------------------------- gate_up
template <int WT, int NCH>
__global__ void __launch_bounds__(kThreads) gateup_kernel(FfnArgs a) {
  extern __shared__ uint4 s_x[];
  constexpr bool kF32 = WT == FT_W_F32;
  constexpr int EPC = W<WT>::kEPC;
  const int H = a.H, I = a.I, k = a.k, T = a.T;
  const int act_bytes = kF32 ? 4 : 2;
  {  // stage x [T][H]
    const int n16 = T * H * act_bytes / 16;
    const uint4* src = static_cast<const uint4*>(a.x);
    for (int i = threadIdx.x; i < n16; i += kThreads) s_x[i] = src[i];
  }
  __syncthreads();
  const int n_u = __ldg(&a.hdr[PH_UNIQUE]);
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.x * (kThreads / 32);
  const int nch = H / EPC;                       // 16-byte chunks per weight row
  const long long row_bytes = (long long)H * W<WT>::kBytes;
  const long long scale_off = 3LL * H * I * W<WT>::kBytes;
  const int sblk = H / 128;                      // fp8: scale blocks per row
  for (int task = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); task < n_u * I; task += warps) {
    const int u = task / I, r = task - u * I;
    const uint8_t* blob = a.pool + (long long)__ldg(&a.unique_slot[u]) * a.expert_bytes;
    const uint8_t* rg = blob + r * row_bytes;
    const uint8_t* ru = blob + (long long)(I + r) * row_bytes;
    const int row0 = __ldg(&a.u_offset[u]);
    const int nrows = min(__ldg(&a.u_offset[u + 1]) - row0, kMaxRows);
    int tok[kMaxRows];
#pragma unroll
    for (int q = 0; q < kMaxRows; ++q) tok[q] = q < nrows ? __ldg(&a.rows_by_u[row0 + q]) / k : 0;
    float ag[kMaxRows], au[kMaxRows];
#pragma unroll
    for (int q = 0; q < kMaxRows; ++q) ag[q] = au[q] = 0.0f;
    for (int c0 = 0; c0 < nch; c0 += 32 * NCH) {
      uint4 wg[NCH], wu[NCH];
#pragma unroll
      for (int i = 0; i < NCH; ++i) {
        const int c = c0 + i * 32 + lane;
        if (c < nch) {
          wg[i] = ldg16(rg + 16LL * c);
          wu[i] = ldg16(ru + 16LL * c);
        }
      }
#pragma unroll
      for (int i = 0; i < NCH; ++i) {
        const int c = c0 + i * 32 + lane;
        if (c < nch) {
          float fg[EPC], fu[EPC];
          decode_chunk<WT>(wg[i], fg);
          decode_chunk<WT>(wu[i], fu);
          float sg = 1.0f, su = 1.0f;
          if (WT == FT_W_FP8E4M3_B128) {
            const int cb = (c * EPC) >> 7;
            sg = scale_at(blob, scale_off, (r >> 7) * sblk + cb);
            su = scale_at(blob, scale_off, (I >> 7) * sblk + (r >> 7) * sblk + cb);
          }
#pragma unroll
          for (int q = 0; q < kMaxRows; ++q) {
            if (q < nrows) {
              float xv[EPC];
              const uint8_t* xrow = reinterpret_cast<const uint8_t*>(s_x) + (long long)tok[q] * H * act_bytes;
              load_act<kF32>(xrow, c * EPC, xv, EPC);
              float pg = 0.0f, pu = 0.0f;
#pragma unroll
              for (int e = 0; e < EPC; ++e) {
                pg = fmaf(fg[e], xv[e], pg);
                pu = fmaf(fu[e], xv[e], pu);
              }
              ag[q] = fmaf(sg, pg, ag[q]);
              au[q] = fmaf(su, pu, au[q]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int q = 0; q < kMaxRows; ++q) {
      if (q < nrows) {
        const float g = warp_sum(ag[q]);
        const float v = warp_sum(au[q]);
        if (lane == 0) a.h[(long long)__ldg(&a.rows_by_u[row0 + q]) * I + r] = g / (1.0f + expf(-g)) * v;
      }
    }
  }
}

// ---------------------------------------------------------------- down
template <int WT, int CPL>
__global__ void __launch_bounds__(kThreads) down_kernel(FfnArgs a) {
  constexpr int EPC = W<WT>::kEPC;
  constexpr int UG = 4;  // experts whose chunks are in flight together
  const int H = a.H, I = a.I, T = a.T;
  const int n_u = __ldg(&a.hdr[PH_UNIQUE]);
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.x * (kThreads / 32);
  const int nch = I / EPC;
  const long long row_bytes = (long long)I * W<WT>::kBytes;
  const long long wd_off = 2LL * H * I * W<WT>::kBytes;
  const long long scale_off = 3LL * H * I * W<WT>::kBytes;
  const int sblk = I / 128;
  const int sbase = 2 * (I / 128) * (H / 128);
  for (int c_out = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); c_out < H; c_out += warps) {
    float acc[kMaxRows];
#pragma unroll
    for (int q = 0; q < kMaxRows; ++q) acc[q] = 0.0f;
    for (int u0 = 0; u0 < n_u; u0 += UG) {
      uint4 w[UG][CPL];
      const uint8_t* blob[UG];
#pragma unroll
      for (int g = 0; g < UG; ++g) {
        blob[g] = nullptr;
        if (u0 + g < n_u) {
          blob[g] = a.pool + (long long)__ldg(&a.unique_slot[u0 + g]) * a.expert_bytes;
          const uint8_t* row = blob[g] + wd_off + c_out * row_bytes;
#pragma unroll
          for (int i = 0; i < CPL; ++i) {
            const int c = i * 32 + lane;
            if (c < nch) w[g][i] = ldg16(row + 16LL * c);
          }
        }
      }
#pragma unroll
      for (int g = 0; g < UG; ++g) {
        if (u0 + g < n_u) {
          const int row0 = __ldg(&a.u_offset[u0 + g]);
          const int nrows = min(__ldg(&a.u_offset[u0 + g + 1]) - row0, kMaxRows);
#pragma unroll
          for (int i = 0; i < CPL; ++i) {
            const int c = i * 32 + lane;
            if (c < nch) {
              float f[EPC];
              decode_chunk<WT>(w[g][i], f);
              float sc = 1.0f;
              if (WT == FT_W_FP8E4M3_B128) sc = scale_at(blob[g], scale_off, sbase + (c_out >> 7) * sblk + ((c * EPC) >> 7));
#pragma unroll
              for (int q = 0; q < kMaxRows; ++q) {
                if (q < nrows) {
                  const int row = __ldg(&a.rows_by_u[row0 + q]);
                  const float4* hp = reinterpret_cast<const float4*>(a.h + (long long)row * I + c * EPC);
                  float p = 0.0f;
#pragma unroll
                  for (int e4 = 0; e4 < EPC / 4; ++e4) {
                    const float4 hv = __ldcg(hp + e4);
                    p = fmaf(f[4 * e4], hv.x, p);
                    p = fmaf(f[4 * e4 + 1], hv.y, p);
                    p = fmaf(f[4 * e4 + 2], hv.z, p);
                    p = fmaf(f[4 * e4 + 3], hv.w, p);
                  }
                  const float wv = __ldg(&a.topk_w[row]) * sc;
                  const int t = row / a.k;
#pragma unroll
                  for (int tt = 0; tt < kMaxRows; ++tt)
                    if (tt == t) acc[tt] = fmaf(wv, p, acc[tt]);
                }
              }
            }
          }
        }
      }
    }
#pragma unroll
    for (int t = 0; t < kMaxRows; ++t) {
      if (t < T) {
        const float v = warp_sum(acc[t]);
        if (lane == 0) static_cast<float*>(a.y)[(long long)t * H + c_out] = v;
      }
    }
  }
}

template <int WT>
cudaError_t gateup_typed(const FfnArgs& a, cudaStream_t s) {
  const int act_bytes = WT == FT_W_F32 ? 4 : 2;
  const size_t xs = (size_t)a.T * a.H * act_bytes;
  const int grid = 152 * 4;
  if (a.H / W<WT>::kEPC <= 64) {
    if (xs > 48 * 1024) cudaFuncSetAttribute(gateup_kernel<WT, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)xs);
    gateup_kernel<WT, 2><<<grid, kThreads, xs, s>>>(a);
  } else {
    if (xs > 48 * 1024) cudaFuncSetAttribute(gateup_kernel<WT, 8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)xs);
    gateup_kernel<WT, 8><<<grid, kThreads, xs, s>>>(a);
  }
  return cudaGetLastError();
}

template <int WT>
cudaError_t down_typed(const FfnArgs& a, cudaStream_t s) {
  const int nch_i = a.I / W<WT>::kEPC;
  const int grid = (a.H + (kThreads / 32) - 1) / (kThreads / 32);
  if (nch_i <= 32)
    down_kernel<WT, 1><<<grid, kThreads, 0, s>>>(a);
  else if (nch_i <= 64)
    down_kernel<WT, 2><<<grid, kThreads, 0, s>>>(a);
  else if (nch_i <= 128)
    down_kernel<WT, 4><<<grid, kThreads, 0, s>>>(a);
  else
    down_kernel<WT, 8><<<grid, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_gateup(const FfnArgs& a, cudaStream_t s) {
  switch (a.wdtype) {
    case FT_W_F32: return gateup_typed<FT_W_F32>(a, s);
    case FT_W_BF16: return gateup_typed<FT_W_BF16>(a, s);
    case FT_W_FP8E4M3_B128: return gateup_typed<FT_W_FP8E4M3_B128>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_down(const FfnArgs& a, cudaStream_t s) {
  switch (a.wdtype) {
    case FT_W_F32: return down_typed<FT_W_F32>(a, s);
    case FT_W_BF16: return down_typed<FT_W_BF16>(a, s);
    case FT_W_FP8E4M3_B128: return down_typed<FT_W_FP8E4M3_B128>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ft
