// Prefill-path expert FFN (T > 8 tokens per layer event), bf16 or fp8 weights: the
// token permutation, the two grouped GEMMs of the routed SwiGLU experts
// (tcgen05 tensor cores, prefill_tc.cu) reading the weights straight from
// their cache slots, and the combine.
//
//   group_rows:  the T*k (token, pick) rows sorted by unique expert (ascending
//                row within an expert): rows_by_u, and pos[row] = its place
//                (a counting sort over chunks of rows: three small kernels)
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

#include <climits>

#include "ft_internal.h"

namespace ft {
namespace {

constexpr int kPThreads = 256;

// ---------------------------------------------------------------- group_rows
// A stable counting sort of the T*k rows by expert, in three passes over
// chunks of kGChunk consecutive rows:
//   chunk_hist:  hist[e][g] = rows of chunk g that picked expert e
//   hist_scan:   hist[e][g] = rows of chunks before g that picked e (one warp
//                per expert)
//   scatter:     each chunk places its rows at u_offset[u(e)] + hist[e][g] +
//                the rows of e before them in the chunk, found 256 rows at a
//                time: a warp's lanes with the same expert rank themselves
//                by lane (__match_any_sync), a shared table counts each
//                warp's rows per expert for the later warps, and a running
//                count per expert carries over to the next 256.
// Rows of an expert end up in ascending row order, as a sort keyed by
// (expert, row) would place them.
constexpr int kGChunk = 512;
constexpr int kGWarps = kPThreads / 32;

__global__ void __launch_bounds__(kPThreads) chunk_hist_kernel(PrefillArgs a, int G) {
  __shared__ int s_h[kMaxExperts];
  const int R = a.T * a.k, g = blockIdx.x;
  for (int e = threadIdx.x; e < a.E; e += kPThreads) s_h[e] = 0;
  __syncthreads();
  for (int r = g * kGChunk + threadIdx.x; r < min(R, (g + 1) * kGChunk); r += kPThreads) {
    const int e = __ldg(&a.topk_idx[r]);
    if (checked_ok(e >= 0 && e < a.E, a.status)) atomicAdd(&s_h[e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < a.E; e += kPThreads) a.hist[(long long)e * G + g] = s_h[e];
}

__global__ void __launch_bounds__(kPThreads) hist_scan_kernel(PrefillArgs a, int G) {
  const int e = blockIdx.x * kGWarps + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (e >= a.E) return;
  int* h = a.hist + (long long)e * G;
  int carry = 0;
  for (int g0 = 0; g0 < G; g0 += 32) {
    const int v = g0 + lane < G ? h[g0 + lane] : 0;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (g0 + lane < G) h[g0 + lane] = carry + x - v;
    carry += __shfl_sync(0xffffffffu, x, 31);
  }
}

__global__ void __launch_bounds__(kPThreads) group_scatter_kernel(PrefillArgs a, int G) {
  __shared__ int s_next[kMaxExperts];          // next place of each expert's rows
  __shared__ int s_wcnt[kGWarps][kMaxExperts];  // rows per (warp, expert) of the current 256
  const int R = a.T * a.k, g = blockIdx.x;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int n_u = min(__ldg(&a.hdr[PH_UNIQUE]), a.E);
  for (int i = threadIdx.x; i < kGWarps * a.E; i += kPThreads) s_wcnt[i / a.E][i % a.E] = 0;
  for (int e = threadIdx.x; e < a.E; e += kPThreads) s_next[e] = INT_MIN / 2;  // an expert outside the plan: p < 0
  __syncthreads();
  for (int u = threadIdx.x; u < n_u; u += kPThreads) {
    const int e = __ldg(&a.unique_expert[u]);
    if (checked_ok(e >= 0 && e < a.E, a.status)) s_next[e] = __ldg(&a.u_offset[u]) + a.hist[(long long)e * G + g];
  }
  __syncthreads();
  const int r_end = min(R, (g + 1) * kGChunk);
  for (int r0 = g * kGChunk; r0 < r_end; r0 += kPThreads) {
    const int r = r0 + threadIdx.x;
    int e = r < r_end ? __ldg(&a.topk_idx[r]) : -1;
    if (e >= a.E) e = -1;  // reported by chunk_hist in the checked build
    const unsigned same = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(same & ((1u << lane) - 1u));
    if (e >= 0 && rank == 0) s_wcnt[w][e] = __popc(same);
    __syncthreads();
    if (e >= 0) {
      int p = s_next[e] + rank;
      for (int q = 0; q < w; ++q) p += s_wcnt[q][e];
      if (checked_ok(p >= 0 && p < R, a.status)) {
        a.rows_by_u[p] = r;
        a.pos[r] = p;
      }
    }
    __syncthreads();  // every thread has read s_next and s_wcnt
    if (e >= 0 && rank == 0) {
      atomicAdd(&s_next[e], __popc(same));
      s_wcnt[w][e] = 0;
    }
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
constexpr int kPermUnroll = 8;  // 16-byte chunks per lane in flight: a 4 KB bf16 row per warp
template <bool kF16>
__global__ void __launch_bounds__(kPThreads) permute_rows_kernel(PrefillArgs a) {
  const int R = a.T * a.k, n16 = a.H / 8;
  const int lane = threadIdx.x & 31;
  const uint4* x = static_cast<const uint4*>(a.x);
  uint4* xp = static_cast<uint4*>(a.xp);
  const int stride = (gridDim.x * kPThreads) >> 5;
  int p = (blockIdx.x * kPThreads + threadIdx.x) >> 5;
  int row_next = p < R ? __ldg(&a.rows_by_u[p]) : 0;
  for (; p < R; p += stride) {
    const int row = row_next;  // the next row's index is in flight while this row moves
    if (p + stride < R) row_next = __ldg(&a.rows_by_u[p + stride]);
    if (!checked_ok(row >= 0 && row < R, a.status)) continue;
    const int t = row / a.k;
    const uint4* src = x + (long long)t * n16;
    uint4* dst = xp + (long long)p * n16;
    for (int i0 = lane; i0 < n16; i0 += 32 * kPermUnroll) {  // a lane's chunks of the row loaded, then stored
      uint4 v[kPermUnroll];
#pragma unroll
      for (int u = 0; u < kPermUnroll; ++u)
        if (i0 + 32 * u < n16) v[u] = __ldg(src + i0 + 32 * u);
#pragma unroll
      for (int u = 0; u < kPermUnroll; ++u)
        if (i0 + 32 * u < n16) {
          if (kF16)
            v[u] = make_uint4(bf16x2_to_f16x2(v[u].x), bf16x2_to_f16x2(v[u].y), bf16x2_to_f16x2(v[u].z),
                              bf16x2_to_f16x2(v[u].w));
          dst[i0 + 32 * u] = v[u];
        }
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

// One full wave of a grid-stride kernel: the CTAs of 256 threads an SM holds
// at once (from its registers and shared memory) times the SMs, so no SM runs
// a partial second wave.
template <typename K>
int full_wave(K kernel) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kPThreads, 0) != cudaSuccess || per_sm < 1)
    per_sm = 4;
  return per_sm * prefill_sms();
}

// The three grids, worked out once per process (the first call comes from
// cache creation, outside any stream capture).
struct PrefillGrids {
  int permute_f16, permute_bf16, combine;
};
const PrefillGrids& prefill_grids() {
  static const PrefillGrids g = {full_wave(permute_rows_kernel<true>), full_wave(permute_rows_kernel<false>),
                                 full_wave(combine_kernel)};
  return g;
}

}  // namespace

void prefill_init() { (void)prefill_grids(); }

int group_chunks(long long rows) { return (int)((rows + kGChunk - 1) / kGChunk); }

bool prefill_supported(int H, int I, int wdtype, int E) {
  return (wdtype == FT_W_BF16 || wdtype == FT_W_FP8E4M3_B128) && prefill_tc_supported(H, I) && E <= kMaxExperts;
}

cudaError_t launch_prefill_ffn(const PrefillArgs& a, int num_slots, cudaStream_t s, int* launches,
                               const cudaEvent_t* marks) {
  const int G = group_chunks(a.T * a.k);
  chunk_hist_kernel<<<G, kPThreads, 0, s>>>(a, G);
  hist_scan_kernel<<<(a.E + kGWarps - 1) / kGWarps, kPThreads, 0, s>>>(a, G);
  group_scatter_kernel<<<G, kPThreads, 0, s>>>(a, G);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (a.wdtype == FT_W_FP8E4M3_B128)
    permute_rows_kernel<true><<<prefill_grids().permute_f16, kPThreads, 0, s>>>(a);
  else
    permute_rows_kernel<false><<<prefill_grids().permute_bf16, kPThreads, 0, s>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = launch_prefill_gemms(a, num_slots, s, marks)) != cudaSuccess) return e;
  combine_kernel<<<prefill_grids().combine, kPThreads, 0, s>>>(a);
  *launches = 7;
  return cudaGetLastError();
}

}  // namespace ft
