// Prefill-path expert FFN (T > 8 tokens per layer event), bf16 or fp8 weights: the
// token permutation, the two grouped GEMMs of the routed SwiGLU experts
// (tcgen05 tensor cores, prefill_tc.cu) reading the weights straight from
// their cache slots, and the combine.
//
//   group_rows:  the T*k (token, pick) rows sorted by unique expert (ascending
//                row within an expert): rows_by_u, and pos[row] = its place
//   permute:     xp[p] = x[t] for the grouped row p of (t, j), so each GEMM
//                tile's A rows are one contiguous block (fp16 for fp8 experts)
//   gate/up:     h[p][i] = silu(Wg[i] . x_t) * (Wu[i] . x_t)  (bf16 h; p the
//                grouped place of row (t, j))
//   down:        yp[p][c] = w_tj * (Wd[c] . h[p])              (fp16; fp32 accumulation)
//   combine:     y[t][c] = sum over j < k, ascending, of yp[pos[t*k+j]][c]
//
// The combine sums each token's picks in a fixed order: the result does not
// depend on how the GEMM tiles were scheduled.
//
// The grouped SwiGLU expert and its gate-weighted combine follow the routed
// experts of the MoE layers the pages serve ("FreeToken vs vLLM on one RTX
// 3090", "Why the performance differs"; the prefill chunk of "FreeToken:
// Efficient Edge-Native MoE Serving ...", ablation paragraph).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ft_internal.h"

namespace ft {
namespace {

constexpr int kPThreads = 256;

// ---------------------------------------------------------------- group_rows
// One CTA per unique expert: its rows in ascending row order, 16 consecutive
// rows per thread per round and one block scan per 4096 rows.
constexpr int kGRows = 16;
__global__ void __launch_bounds__(kPThreads) group_rows_kernel(PrefillArgs a) {
  __shared__ int s_warp[kPThreads / 32];
  const int n_u = __ldg(&a.hdr[PH_UNIQUE]);
  const int u = blockIdx.x;
  if (u >= n_u) return;
  const int e = __ldg(&a.unique_expert[u]);
  const int rows = a.T * a.k;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int carry = __ldg(&a.u_offset[u]);
  for (int base = 0; base < rows; base += kPThreads * kGRows) {
    const int r0 = base + threadIdx.x * kGRows;
    int idx[kGRows];
    int cnt = 0;
#pragma unroll
    for (int i = 0; i < kGRows; ++i) {
      idx[i] = r0 + i < rows ? __ldg(&a.topk_idx[r0 + i]) : -1;
      cnt += idx[i] == e;
    }
    int x = cnt;  // inclusive warp scan, then across warps
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[w] = x;
    __syncthreads();
    int before = 0, total = 0;
#pragma unroll
    for (int q = 0; q < kPThreads / 32; ++q) {
      before += q < w ? s_warp[q] : 0;
      total += s_warp[q];
    }
    int p = carry + before + x - cnt;
#pragma unroll
    for (int i = 0; i < kGRows; ++i)
      if (idx[i] == e && checked_ok(p >= 0 && p < rows, a.status)) {
        a.rows_by_u[p] = r0 + i;
        a.pos[r0 + i] = p;
        ++p;
      }
    carry += total;
    __syncthreads();
  }
}

// ---------------------------------------------------------------- permute
// One warp per grouped row: xp[p] = x[rows_by_u[p] / k], 16-byte chunks; for
// fp8 experts (whose GEMMs multiply fp16 operands) the bf16 values are
// converted to fp16 on the way.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
  const __half2 h = __floats2half2_rn(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
  return *reinterpret_cast<const uint32_t*>(&h);
}
template <bool kF16>
__global__ void __launch_bounds__(kPThreads) permute_rows_kernel(PrefillArgs a) {
  const int R = a.T * a.k, n16 = a.H / 8;
  const int lane = threadIdx.x & 31;
  const uint4* x = static_cast<const uint4*>(a.x);
  uint4* xp = static_cast<uint4*>(a.xp);
  for (int p = (blockIdx.x * kPThreads + threadIdx.x) >> 5; p < R; p += (gridDim.x * kPThreads) >> 5) {
    const int row = __ldg(&a.rows_by_u[p]);
    if (!checked_ok(row >= 0 && row < R, a.status)) continue;
    const int t = row / a.k;
    const uint4* src = x + (long long)t * n16;
    uint4* dst = xp + (long long)p * n16;
    for (int i = lane; i < n16; i += 32) {
      uint4 v = __ldg(src + i);
      if (kF16) v = make_uint4(bf16x2_to_f16x2(v.x), bf16x2_to_f16x2(v.y), bf16x2_to_f16x2(v.z), bf16x2_to_f16x2(v.w));
      dst[i] = v;
    }
  }
}

// ---------------------------------------------------------------- combine
// y[t][c] = sum_{j<k} yp[pos[t*k+j]][c] in fp32, four columns per thread.
__global__ void __launch_bounds__(kPThreads) combine_kernel(PrefillArgs a) {
  const int q4 = a.H / 4;
  const long long n = (long long)a.T * q4;
  for (long long i = (long long)blockIdx.x * kPThreads + threadIdx.x; i < n; i += (long long)gridDim.x * kPThreads) {
    const int t = (int)(i / q4), q = (int)(i - (long long)t * q4);
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < a.k; ++j) {
      const int p = __ldg(&a.pos[t * a.k + j]);
      if (!checked_ok(p >= 0 && p < a.T * a.k, a.status)) continue;
      const uint2 v = __ldcg(reinterpret_cast<const uint2*>(static_cast<const __half*>(a.yp) + (long long)p * a.H) + q);
      const float2 lo = __half22float2(*reinterpret_cast<const __half2*>(&v.x));
      const float2 hi = __half22float2(*reinterpret_cast<const __half2*>(&v.y));
      s.x += lo.x; s.y += lo.y; s.z += hi.x; s.w += hi.y;
    }
    reinterpret_cast<float4*>(a.y + (long long)t * a.H)[q] = s;
  }
}

int prefill_sms() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
  }
  return n;
}

}  // namespace

bool prefill_supported(int H, int I, int wdtype, int E) {
  return (wdtype == FT_W_BF16 || wdtype == FT_W_FP8E4M3_B128) && prefill_tc_supported(H, I) && E <= kMaxExperts;
}

cudaError_t launch_prefill_ffn(const PrefillArgs& a, int num_slots, cudaStream_t s, int* launches,
                               const cudaEvent_t* marks) {
  group_rows_kernel<<<a.E, kPThreads, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (a.wdtype == FT_W_FP8E4M3_B128)
    permute_rows_kernel<true><<<8 * prefill_sms(), kPThreads, 0, s>>>(a);
  else
    permute_rows_kernel<false><<<8 * prefill_sms(), kPThreads, 0, s>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = launch_prefill_gemms(a, num_slots, s, marks)) != cudaSuccess) return e;
  combine_kernel<<<4 * prefill_sms(), kPThreads, 0, s>>>(a);
  *launches = 5;
  return cudaGetLastError();
}

}  // namespace ft
