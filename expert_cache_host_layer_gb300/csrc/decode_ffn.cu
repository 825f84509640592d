// Decode-path expert FFN (T <= 8 tokens): two HBM-bound kernels that stream
// the expert weights straight from their cache slots through shared memory.
//
//   gate_up:  h[row][r] = silu(Wg[r] . x_t) * (Wu[r] . x_t)   for every row
//             (t, j) of every unique expert u and every r < I
//   down:     y[t][c]  = sum_u sum_(rows (t,j) of u) w_tj * (Wd[c] . h[row])   (fp32 y)
//
// Both kernels are warp-specialised pipelines: one producer thread issues
// bulk asynchronous copies (cp.async.bulk, completion counted on an
// mbarrier) of contiguous weight-row blocks into a ring of shared-memory
// stages, and eight consumer warps take one weight row each per stage.  A
// gate_up work unit is (expert u, P row pairs): the Wg rows and the Wu rows of
// the unit are each one contiguous block of the slot.  A down work unit is a
// block of 8 output columns c, streamed expert by expert; the combine over
// experts happens in registers in ascending expert order, with no atomics.
// The down kernel is launched as a programmatic dependent of gate_up: its
// producer starts streaming Wd while gate_up finishes, and its consumers wait
// for gate_up's h (griddepcontrol.wait) before reading it.
//
// Every mbarrier wait is bounded (about one second of %globaltimer); a wait
// that runs out records FT_ERR_TIMEOUT in the status word.  The producer then
// stops issuing; a consumer stops waiting but runs its loop to the end (its
// results are garbage), so every consumer warp still reaches each named
// barrier and the kernel ends instead of hanging.
//
// The SwiGLU expert and the gate-weighted combine follow the routed experts
// of the Qwen3-MoE / DeepSeek MoE layers the pages serve ("FreeToken vs vLLM
// on one RTX 3090", "Why the performance differs"; "FreeToken: Efficient
// Edge-Native MoE Serving ...", design paragraph: the FFN reads experts from
// the GPU expert cache).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <map>
#include <mutex>
#include <utility>

#include "ft_internal.h"

namespace ft {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;  // + one producer warp
constexpr int kMaxRows = kDecodeMaxTokens;           // rows of one expert in a decode batch
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
__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory"); }
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


// Shared-memory layouts (bytes), shared by the kernels and their launchers.
// Plan staged in shared memory: unique_slot[n], u_offset[n+1], rows_by_u[rows].
__host__ __device__ __forceinline__ int plan_bytes(int max_unique, int rows) {
  return (2 * max_unique + 1 + rows) * 4;
}

struct GateUpLayout {
  int P, NS, stage_bytes, x_off, res_off, plan_off, bar_off, total;
  __host__ __device__ GateUpLayout(int H, int I, int T, int wsize, int act_bytes, int max_unique, int rows) {
    int p = 16384 / (H * wsize);  // rows of one matrix per unit: about 16 KB per matrix
    if (p < 1) p = 1;
    P = 1;
    while (P * 2 <= p && I % (P * 2) == 0) P *= 2;
    stage_bytes = 2 * P * H * wsize;
    NS = stage_bytes <= 16384 ? 6 : 3;
    x_off = NS * stage_bytes;
    res_off = align_up(x_off + T * H * act_bytes, 16);
    plan_off = align_up(res_off + 2 * 2 * P * kMaxRows * 4, 16);
    bar_off = align_up(plan_off + plan_bytes(max_unique, rows), 16);
    total = bar_off + 2 * NS * 8;
  }
};
struct DownLayout {
  int RD, NS, stage_bytes, h_off, h_bytes, plan_off, bar_off, total;
  __host__ __device__ DownLayout(int I, int wsize, int max_unique, int rows) {
    RD = kConsumerWarps;  // one output column per consumer warp
    stage_bytes = RD * I * wsize;
    NS = stage_bytes <= 8192 ? 8 : 6;
    h_off = NS * stage_bytes;
    h_bytes = rows * I * 4;
    if (h_bytes > 64 * 1024) h_bytes = 0;  // large batches read h from L2 instead
    plan_off = align_up(h_off + h_bytes, 16);
    bar_off = align_up(plan_off + plan_bytes(max_unique, rows), 16);
    total = bar_off + 2 * NS * 8;
  }
};

// Copies the plan arrays the FFN kernels index into shared memory.
__device__ __forceinline__ void stage_plan(const FfnArgs& a, int n_u, int32_t* s_slot, int32_t* s_off,
                                           int32_t* s_rows) {
  const int rows = a.T * a.k;
  for (int i = threadIdx.x; i < n_u; i += blockDim.x) s_slot[i] = __ldg(&a.unique_slot[i]);
  for (int i = threadIdx.x; i <= n_u; i += blockDim.x) s_off[i] = __ldg(&a.u_offset[i]);
  for (int i = threadIdx.x; i < rows; i += blockDim.x) s_rows[i] = __ldg(&a.rows_by_u[i]);
}

// ---------------------------------------------------------------- gate_up
template <int WT>
__global__ void __launch_bounds__(kThreads, 2) gateup_kernel(FfnArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr bool kF32 = WT == FT_W_F32;
  constexpr int EPC = W<WT>::kEPC, WSZ = W<WT>::kBytes;
  const int H = a.H, I = a.I, k = a.k, T = a.T;
  const int act_bytes = kF32 ? 4 : 2;
  const GateUpLayout lay(H, I, T, WSZ, act_bytes, a.max_unique, T * k);
  const int P = lay.P, NS = lay.NS;
  uint8_t* xs = smem + lay.x_off;
  float* res = reinterpret_cast<float*>(smem + lay.res_off);
  int32_t* p_slot = reinterpret_cast<int32_t*>(smem + lay.plan_off);
  int32_t* p_off = p_slot + a.max_unique;
  int32_t* p_rows = p_off + a.max_unique + 1;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + lay.bar_off);
  uint64_t* empty = full + NS;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_u = min(__ldg(&a.hdr[PH_UNIQUE]), a.max_unique);

  if (threadIdx.x == 0) {
    wait_ready_flag(a);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    mbar_init_fence();
  }
  {  // stage x [T][H]
    const int n16 = T * H * act_bytes / 16;
    const uint4* src = static_cast<const uint4*>(a.x);
    for (int i = threadIdx.x; i < n16; i += kThreads) reinterpret_cast<uint4*>(xs)[i] = src[i];
  }
  stage_plan(a, n_u, p_slot, p_off, p_rows);
  __syncthreads();
  pdl_launch_dependents();  // the down kernel may start streaming Wd now

  const int units_per_u = I / P;
  const int n_units = n_u * units_per_u;
  const long long row_bytes = (long long)H * WSZ;
  const uint32_t block_bytes = (uint32_t)(P * row_bytes);

  if (warp == kConsumerWarps) {  // producer
    if (lane == 0) {
      int it = 0;
      for (int unit = blockIdx.x; unit < n_units; unit += gridDim.x, ++it) {
        const int s = it % NS;
        if (it >= NS && !mbar_wait(&empty[s], ((it / NS) & 1) ^ 1, a.status)) break;
        const int u = unit / units_per_u, pb = unit - u * units_per_u;
        const uint8_t* blob = a.pool + (long long)p_slot[u] * a.expert_bytes;
        uint8_t* st = smem + (size_t)s * lay.stage_bytes;
        mbar_expect_tx(&full[s], 2 * block_bytes);
        bulk_g2s(st, blob + (long long)pb * P * row_bytes, block_bytes, &full[s]);
        bulk_g2s(st + block_bytes, blob + (long long)(I + pb * P) * row_bytes, block_bytes, &full[s]);
      }
    }
    return;
  }

  // consumers: warp w takes rows w, w+8, ... of the stage's 2P rows (Wg rows, then Wu rows)
  const int nch = H / EPC;
  const long long scale_off = 3LL * H * I * WSZ;
  const int sblk = H / 128;
  int it = 0, buf = 0;
  bool aborted = false;
  for (int unit = blockIdx.x; unit < n_units; unit += gridDim.x, ++it) {
    const int s = it % NS;
    const int u = unit / units_per_u, pb = unit - u * units_per_u;
    const int row0 = p_off[u];
    const int nrows = min(p_off[u + 1] - row0, kMaxRows);
    int tok[kMaxRows];
#pragma unroll
    for (int q = 0; q < kMaxRows; ++q) tok[q] = q < nrows ? p_rows[row0 + q] / k : 0;
    const uint8_t* blob = a.pool + (long long)p_slot[u] * a.expert_bytes;
    if (!aborted && !mbar_wait(&full[s], (it / NS) & 1, a.status)) aborted = true;
    const uint8_t* st = smem + (size_t)s * lay.stage_bytes;
    for (int rr = warp; rr < 2 * P; rr += kConsumerWarps) {
      const bool is_up = rr >= P;
      const int r = pb * P + (is_up ? rr - P : rr);  // row within its matrix
      const uint4* wrow = reinterpret_cast<const uint4*>(st + (size_t)rr * row_bytes);
      float acc[kMaxRows];
#pragma unroll
      for (int q = 0; q < kMaxRows; ++q) acc[q] = 0.0f;
      for (int c = lane; c < nch; c += 32) {
        float f[EPC];
        decode_chunk<WT>(wrow[c], f);
        float sc = 1.0f;
        if (WT == FT_W_FP8E4M3_B128)
          sc = scale_at(blob, scale_off, (is_up ? (I >> 7) * sblk : 0) + (r >> 7) * sblk + ((c * EPC) >> 7));
#pragma unroll
        for (int q = 0; q < kMaxRows; ++q) {
          if (q < nrows) {
            float xv[EPC];
            load_act<kF32, EPC>(xs + (size_t)tok[q] * H * act_bytes, c * EPC, xv);
            float p = 0.0f;
#pragma unroll
            for (int e = 0; e < EPC; ++e) p = fmaf(f[e], xv[e], p);
            acc[q] = fmaf(sc, p, acc[q]);
          }
        }
      }
#pragma unroll
      for (int q = 0; q < kMaxRows; ++q) {
        if (q < nrows) {
          const float v = warp_sum(acc[q]);
          if (lane == 0) res[(buf * 2 * P + rr) * kMaxRows + q] = v;
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);  // this warp is done reading the stage
    consumer_sync();
    for (int i = threadIdx.x; i < P * nrows; i += kConsumerWarps * 32) {
      const int p = i / nrows, q = i - p * nrows;
      const float g = res[(buf * 2 * P + p) * kMaxRows + q];
      const float v = res[(buf * 2 * P + P + p) * kMaxRows + q];
      const int row = p_rows[row0 + q];
      a.h[(long long)row * I + pb * P + p] = g / (1.0f + expf(-g)) * v;
    }
    buf ^= 1;
  }
}

// ---------------------------------------------------------------- down
template <int WT>
__global__ void __launch_bounds__(kThreads, 2) down_kernel(FfnArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int EPC = W<WT>::kEPC, WSZ = W<WT>::kBytes;
  const int H = a.H, I = a.I, T = a.T, k = a.k;
  const DownLayout lay(I, WSZ, a.max_unique, T * k);
  const int RD = lay.RD, NS = lay.NS;
  float* hs = reinterpret_cast<float*>(smem + lay.h_off);
  int32_t* p_slot = reinterpret_cast<int32_t*>(smem + lay.plan_off);
  int32_t* p_off = p_slot + a.max_unique;
  int32_t* p_rows = p_off + a.max_unique + 1;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + lay.bar_off);
  uint64_t* empty = full + NS;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the plan was written by route_classify, which completed before the primary kernel started
  const int n_u = min(__ldg(&a.hdr[PH_UNIQUE]), a.max_unique);
  if (threadIdx.x == 0) {
    wait_ready_flag(a);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    mbar_init_fence();
  }
  stage_plan(a, n_u, p_slot, p_off, p_rows);
  __syncthreads();
  const int n_rb = H / RD;
  const long long row_bytes = (long long)I * WSZ;
  const uint32_t stage_bytes = (uint32_t)(RD * row_bytes);
  const long long wd_off = 2LL * H * I * WSZ;

  if (warp == kConsumerWarps) {  // producer: Wd does not depend on the primary kernel
    if (lane == 0) {
      int it = 0;
      for (int rb = blockIdx.x; rb < n_rb; rb += gridDim.x)
        for (int u = 0; u < n_u; ++u, ++it) {
          const int s = it % NS;
          if (it >= NS && !mbar_wait(&empty[s], ((it / NS) & 1) ^ 1, a.status)) return;
          const uint8_t* blob = a.pool + (long long)p_slot[u] * a.expert_bytes;
          mbar_expect_tx(&full[s], stage_bytes);
          bulk_g2s(smem + (size_t)s * lay.stage_bytes, blob + wd_off + (long long)rb * RD * row_bytes, stage_bytes,
                   &full[s]);
        }
    }
    return;
  }

  pdl_wait_primary();  // h is complete and visible
  const bool h_in_smem = lay.h_bytes > 0;
  if (h_in_smem) {  // consumers copy h [rows][I] once
    const int n4 = T * k * I / 4;
    const float4* src = reinterpret_cast<const float4*>(a.h);
    for (int i = threadIdx.x; i < n4; i += kConsumerWarps * 32) reinterpret_cast<float4*>(hs)[i] = src[i];
    consumer_sync();
  }
  const float* hbase = h_in_smem ? hs : a.h;
  const int nch = I / EPC;
  const long long scale_off = 3LL * H * I * WSZ;
  const int sblk = I / 128;
  const int sbase = 2 * (I / 128) * (H / 128);
  int it = 0;
  bool aborted = false;
  for (int rb = blockIdx.x; rb < n_rb; rb += gridDim.x) {
    const int c_out = rb * RD + warp;  // RD == kConsumerWarps: one column per warp
    float acc[kMaxRows];
#pragma unroll
    for (int q = 0; q < kMaxRows; ++q) acc[q] = 0.0f;
    for (int u = 0; u < n_u; ++u, ++it) {
      const int s = it % NS;
      const int row0 = p_off[u];
      const int nrows = min(p_off[u + 1] - row0, kMaxRows);
      const uint8_t* blob = a.pool + (long long)p_slot[u] * a.expert_bytes;
      int rows[kMaxRows];
      float wts[kMaxRows];
#pragma unroll
      for (int q = 0; q < kMaxRows; ++q) {
        rows[q] = q < nrows ? p_rows[row0 + q] : 0;
        wts[q] = q < nrows ? __ldg(&a.topk_w[rows[q]]) : 0.0f;
      }
      if (!aborted && !mbar_wait(&full[s], (it / NS) & 1, a.status)) aborted = true;
      const uint4* wrow = reinterpret_cast<const uint4*>(smem + (size_t)s * lay.stage_bytes + (size_t)warp * row_bytes);
      float part[kMaxRows];
#pragma unroll
      for (int q = 0; q < kMaxRows; ++q) part[q] = 0.0f;
      for (int c = lane; c < nch; c += 32) {
        float f[EPC];
        decode_chunk<WT>(wrow[c], f);
        float sc = 1.0f;
        if (WT == FT_W_FP8E4M3_B128) sc = scale_at(blob, scale_off, sbase + (c_out >> 7) * sblk + ((c * EPC) >> 7));
#pragma unroll
        for (int q = 0; q < kMaxRows; ++q) {
          if (q < nrows) {
            const float4* hp = reinterpret_cast<const float4*>(hbase + (long long)rows[q] * I + c * EPC);
            float p = 0.0f;
#pragma unroll
            for (int e4 = 0; e4 < EPC / 4; ++e4) {
              const float4 hv = hp[e4];
              p = fmaf(f[4 * e4], hv.x, p);
              p = fmaf(f[4 * e4 + 1], hv.y, p);
              p = fmaf(f[4 * e4 + 2], hv.z, p);
              p = fmaf(f[4 * e4 + 3], hv.w, p);
            }
            part[q] = fmaf(sc, p, part[q]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
#pragma unroll
      for (int q = 0; q < kMaxRows; ++q) {
        if (q < nrows) {
          const int t = rows[q] / k;
#pragma unroll
          for (int tt = 0; tt < kMaxRows; ++tt)
            if (tt == t) acc[tt] = fmaf(wts[q], part[q], acc[tt]);
        }
      }
    }
#pragma unroll
    for (int t = 0; t < kMaxRows; ++t) {
      if (t < T) {
        const float v = warp_sum(acc[t]);
        if (lane == 0) a.y[(long long)t * H + c_out] = v;
      }
    }
  }
}

// ---------------------------------------------------------------- fused
// One CTA per SM, all co-resident (cooperative launch): eight consumer warps
// and one producer warp.
//  producer: one thread (after the copy-engine ready flag, if any) prefetches
//            this CTA's Wd rows of every expert into L2, then streams the
//            CTA's work through a ring of shared-memory stages with bulk
//            asynchronous copies (completion counted on one mbarrier per
//            stage; consumers free a stage through a second mbarrier);
//  phase 1:  the CTA owns a contiguous run of (expert, intermediate row)
//            pairs; a unit is R consecutive rows of one expert: its R Wg
//            rows then its R Wu rows, two contiguous blocks of the slot.
//            Two groups of four warps take alternate units; warp j of a
//            group takes row pairs j, j+4, ...: it dots the Wg row and the Wu
//            row with every token of the expert (one pass over x for both)
//            and writes h = silu(g) * u itself, so units need no CTA-wide
//            synchronisation;
//  barrier:  grid-wide (bounded), h complete everywhere;
//  phase 2:  the CTA owns output columns [c0, c1), cut into pieces of at
//            most PR rows; a unit is one piece of as many experts' Wd as fit
//            in a stage (rows c of Wd are contiguous), pieces outer, experts
//            inner (ascending), so at this shape the whole of a CTA's Wd is
//            in shared memory before the grid barrier is passed.  The
//            column c always belongs to warp (c - piece start) % 8, which
//            keeps its sum over experts in registers and writes y once.
//  copy:     in SM-pull mode up to four more warps copy the NEXT event's missed
//            blobs from the host bank into their victim slots meanwhile (8 KB
//            items spread over all CTAs, 8 loads in flight per thread).  The
//            victims exclude this event's slots (pin rule) and the FFN before
//            this one has finished, so nothing still reads them; the next FFN
//            runs after this kernel on the same stream.  One kernel per layer
//            thus moves the next layer's experts over the host link while
//            this layer's experts stream from HBM.
// Every mbarrier wait is bounded; a wait that runs out records
// FT_ERR_TIMEOUT, sets a CTA-wide abort flag that ends all later waits at
// once, and the producer still waits (bounded) for its copies in flight
// before it exits.
constexpr int kFConsumers = 8;
constexpr int kFCopyWarps = kMaxFetchWarps;  // warps kFConsumers + 1 .. : the next event's miss fetch
constexpr int kFThreads = (kFConsumers + 1 + kFCopyWarps) * 32;
constexpr int kFCopyUnroll = 8;  // 16-byte loads in flight per copy thread
constexpr int kFusedSmemBudget = 150 * 1024;
constexpr int kFStages = 4;
constexpr int kFStageMax = 32 * 1024;
constexpr int kFMaxUnitRows = 32;   // R (row pairs of a phase-1 unit)
constexpr int kFMaxPieceRows = 16;  // PR (Wd rows of a phase-2 unit): two per warp

struct FusedLayout {
  int x_off, plan_off, w_off, bar_off, h_off, h_bytes, ring_off, stage_bytes, R, PR, total;
  __host__ __device__ FusedLayout(int H, int I, int T, int wsize, int act_bytes, int max_unique, int rows) {
    const int row_g = H * wsize, row_d = I * wsize;
    x_off = 0;
    plan_off = align_up(T * H * act_bytes, 128);
    w_off = plan_off + align_up(plan_bytes(max_unique, rows), 16);
    bar_off = w_off + align_up(rows * 4, 16);
    h_off = bar_off + align_up((2 * kFStages + 1) * 8, 128);  // full[], empty[], abort word
    const int fixed = h_off;
    h_bytes = rows * I * 4;
    // h sits in shared memory only if that leaves at least 64 KB of ring
    if (kFusedSmemBudget - fixed - h_bytes < 64 * 1024) h_bytes = 0;
    ring_off = align_up(h_off + h_bytes, 128);
    int sb = (kFusedSmemBudget - ring_off) / kFStages;
    if (sb > kFStageMax) sb = kFStageMax;
    stage_bytes = sb / 128 * 128;
    R = row_g > 0 ? stage_bytes / (2 * row_g) : 0;
    if (R > kFMaxUnitRows) R = kFMaxUnitRows;
    PR = row_d > 0 ? stage_bytes / row_d : 0;
    if (PR > kFMaxPieceRows) PR = kFMaxPieceRows;
    total = ring_off + kFStages * stage_bytes;
  }
  __host__ __device__ bool ok() const { return stage_bytes > 0 && R >= 1 && PR >= 1; }
};

__device__ __forceinline__ uint4 ld_host16(const uint4* p) {  // streamed once: evict first
  uint4 v;
  asm volatile("ld.global.cs.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// The copy warps' work: 16-byte words of the next event's missed blobs, in
// items of nw * 32 * kFCopyUnroll words (nw copy warps take part), item i on
// CTA i % grid.
__device__ __forceinline__ void fused_fetch(const PullArgs& p, int ct, int nw) {
  const long long kItem16 = (long long)nw * 32 * kFCopyUnroll;
  const int n_miss = __ldcg(&p.hdr[PH_MISS]);
  const long long eb16 = p.expert_bytes >> 4;
  const long long per_blob = (eb16 + kItem16 - 1) / kItem16;
  const long long items = (long long)n_miss * per_blob;
  const uint4* bank = static_cast<const uint4*>(p.bank);
  uint4* pool = static_cast<uint4*>(p.pool);
  for (long long it = blockIdx.x; it < items; it += gridDim.x) {
    const int m = (int)(it / per_blob);
    const long long c = it - (long long)m * per_blob;
    const int e = __ldcg(&p.miss_expert[m]);
    const int slot = __ldcg(&p.miss_slot[m]);
    const long long blob = ((long long)p.layer * p.E + e) % p.bank_blobs;
    const uint4* src = bank + blob * eb16 + c * kItem16;
    uint4* dst = pool + (long long)slot * eb16 + c * kItem16;
    const long long n = min(kItem16, eb16 - c * kItem16);
    uint4 v[kFCopyUnroll];
#pragma unroll
    for (int u = 0; u < kFCopyUnroll; ++u) {
      const long long i = (long long)u * (nw * 32) + ct;
      if (i < n) v[u] = ld_host16(src + i);
    }
#pragma unroll
    for (int u = 0; u < kFCopyUnroll; ++u) {
      const long long i = (long long)u * (nw * 32) + ct;
      if (i < n) dst[i] = v[u];
    }
  }
}

__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Bounded mbarrier wait that gives up at once when the CTA has aborted, and
// aborts the CTA when it runs out.
__device__ __forceinline__ bool fwait(uint64_t* bar, uint32_t parity, int32_t* status, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (;;) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_ns() - t0 > kWaitLimitNs) {
      if (status) atomicCAS(status, 0, (int)FT_ERR_TIMEOUT);
      *abort_flag = 1;
      return false;
    }
  }
}

// Consumer-side acquire of a ring stage: lane 0 waits, then every lane
// observes the completed phase itself (so the async-proxy writes are visible
// to it).
__device__ __forceinline__ bool stage_acquire(uint64_t* full, uint32_t parity, int32_t* status,
                                              volatile int* abort_flag) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = fwait(full, parity, status, abort_flag);
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok) mbar_try_wait(full, parity);
  return ok;
}

__device__ __forceinline__ void stage_release(uint64_t* empty) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(empty);
}

__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 2, %0;" ::"n"(kFConsumers * 32) : "memory");
}

// MR: most rows (tokens) of one expert, 1 for single-token decode.
// Phase 2 of the fused kernel for one CTA: y[t][c] for c in [c0, c1).
// kHs: h was copied into shared memory; DCL: 16-byte chunks per lane of one
// Wd row (row bytes = 512 * DCL).  Units continue the ring sequence at `unit`.
template <int WT, int MR, int DCL, bool kHs>
__device__ __forceinline__ void fused_phase2(const FfnArgs& a, const FusedLayout& lay, uint8_t* ring,
                                             uint64_t* full, uint64_t* empty, volatile int* abort_flag,
                                             const int32_t* p_slot, const int32_t* p_off, const int32_t* p_rows,
                                             const float* p_w, const float* hbase, int n_u, int c0, int c1,
                                             int unit) {
  constexpr int EPC = W<WT>::kEPC, WSZ = W<WT>::kBytes;
  const int H = a.H, I = a.I, k = a.k, T = a.T;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int SB = lay.stage_bytes;
  const long long row_d = (long long)I * WSZ, scale_off = 3LL * H * I * WSZ;
  const int sblk = I / 128;
  const int sbase = 2 * (I / 128) * (H / 128);
  for (int p0 = c0; p0 < c1; p0 += lay.PR) {
    const int PR = min(lay.PR, c1 - p0);
    const int EU = max(1, SB / (int)(PR * row_d));  // experts per unit (as the producer packs them)
    float acc[2][MR];
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int t = 0; t < MR; ++t) acc[m][t] = 0.0f;
    for (int ub = 0; ub < n_u; ub += EU, ++unit) {
      const int s = unit % kFStages;
      const bool ok = stage_acquire(&full[s], (unit / kFStages) & 1, a.status, abort_flag);
      const int ne = ok ? min(EU, n_u - ub) : 0;
#pragma unroll 2
      for (int k2 = 0; k2 < ne; ++k2) {
        const int u = ub + k2;
        const int row0 = p_off[u];
        const int nrows = min(p_off[u + 1] - row0, MR);
        int hrow[MR], tok[MR];
        float wgt[MR];
#pragma unroll
        for (int t = 0; t < MR; ++t) {
          const int row = t < nrows ? p_rows[row0 + t] : 0;
          hrow[t] = row * I;
          tok[t] = row / k;
          wgt[t] = t < nrows ? p_w[row] : 0.0f;
        }
        const uint8_t* blob = a.pool + (long long)p_slot[u] * a.expert_bytes;
        const uint8_t* piece = ring + (size_t)s * SB + (size_t)k2 * PR * row_d;
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          const int j = warp + m * kFConsumers;
          if (j < PR) {
            const int cc = p0 + j;
            const uint4* wrow = reinterpret_cast<const uint4*>(piece + j * row_d);
            float part[MR];
#pragma unroll
            for (int t = 0; t < MR; ++t) part[t] = 0.0f;
#pragma unroll
            for (int i = 0; i < DCL; ++i) {
              const int c = i * 32 + lane;
              float f[EPC];
              decode_chunk<WT>(wrow[c], f);
              float sc = 1.0f;
              if (WT == FT_W_FP8E4M3_B128) sc = scale_at(blob, scale_off, sbase + (cc >> 7) * sblk + ((c * EPC) >> 7));
#pragma unroll
              for (int t = 0; t < MR; ++t) {
                if (t < nrows) {
                  const float4* hp = reinterpret_cast<const float4*>(hbase + hrow[t] + c * EPC);
                  float q0 = 0.0f, q1 = 0.0f;
#pragma unroll
                  for (int e4 = 0; e4 < EPC / 4; ++e4) {
                    const float4 hv = kHs ? hp[e4] : __ldcg(hp + e4);
                    q0 = fmaf(f[4 * e4], hv.x, q0);
                    q1 = fmaf(f[4 * e4 + 1], hv.y, q1);
                    q0 = fmaf(f[4 * e4 + 2], hv.z, q0);
                    q1 = fmaf(f[4 * e4 + 3], hv.w, q1);
                  }
                  part[t] = fmaf(sc, q0 + q1, part[t]);
                }
              }
            }
#pragma unroll
            for (int t = 0; t < MR; ++t)  // per-lane partial sums; reduced once per column
              if (t < nrows)
#pragma unroll
                for (int tt = 0; tt < MR; ++tt)
                  if (tt == tok[t]) acc[m][tt] = fmaf(wgt[t], part[t], acc[m][tt]);
          }
        }
      }
      stage_release(&empty[s]);
    }
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      const int j = warp + m * kFConsumers;
      if (j < PR) {
#pragma unroll
        for (int t = 0; t < MR; ++t) {
          if (t < T) {
            const float v = warp_sum(acc[m][t]);
            if (lane == 0) a.y[(long long)t * H + p0 + j] = v;
          }
        }
      }
    }
  }
}

// NCL: 16-byte chunks per lane of one Wg/Wu row (row bytes <= 512 * NCL);
// DCL: the same for one Wd row (row bytes = 512 * DCL).
template <int WT, int MR, int NCL, int DCL>
__global__ void __maxnreg__(96) ffn_fused_kernel(FfnArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr bool kF32 = WT == FT_W_F32;
  constexpr int EPC = W<WT>::kEPC, WSZ = W<WT>::kBytes;
  const int H = a.H, I = a.I, k = a.k, T = a.T;
  const int act_bytes = kF32 ? 4 : 2;
  const int rows_total = T * k;
  const FusedLayout lay(H, I, T, WSZ, act_bytes, a.max_unique, rows_total);
  const uint8_t* xs = smem + lay.x_off;
  int32_t* p_slot = reinterpret_cast<int32_t*>(smem + lay.plan_off);
  int32_t* p_off = p_slot + a.max_unique;
  int32_t* p_rows = p_off + a.max_unique + 1;
  float* p_w = reinterpret_cast<float*>(smem + lay.w_off);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + lay.bar_off);
  uint64_t* empty = full + kFStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kFStages);
  float* hs = reinterpret_cast<float*>(smem + lay.h_off);
  uint8_t* ring = smem + lay.ring_off;
  const int SB = lay.stage_bytes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_u = min(__ldg(&a.hdr[PH_UNIQUE]), a.max_unique);
  const long long row_g = (long long)H * WSZ, row_d = (long long)I * WSZ;
  const long long wd_off = 2LL * H * I * WSZ, scale_off = 3LL * H * I * WSZ;
  // phase-1 rows [q0, q1) of the flattened (expert, intermediate row) index
  const long long nq = (long long)n_u * I;
  const int q0 = (int)(nq * blockIdx.x / gridDim.x), q1 = (int)(nq * (blockIdx.x + 1) / gridDim.x);
  // phase-2 output columns [c0, c1)
  const int c0 = (int)((long long)H * blockIdx.x / gridDim.x);
  const int c1 = (int)((long long)H * (blockIdx.x + 1) / gridDim.x);

  // ---- prologue (all threads): barriers, plan and x into shared memory
  if (threadIdx.x == 0) {
    for (int s = 0; s < kFStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kFConsumers);
    }
    *abort_flag = 0;
    mbar_init_fence();
  }
  for (int i = threadIdx.x; i < n_u; i += kFThreads) p_slot[i] = __ldg(&a.unique_slot[i]);
  for (int i = threadIdx.x; i <= n_u; i += kFThreads) p_off[i] = __ldg(&a.u_offset[i]);
  for (int i = threadIdx.x; i < rows_total; i += kFThreads) {
    p_rows[i] = __ldg(&a.rows_by_u[i]);
    p_w[i] = __ldg(&a.topk_w[i]);
  }
  {
    const int n16 = T * H * act_bytes / 16;
    const uint4* src = static_cast<const uint4*>(a.x);
    for (int i = threadIdx.x; i < n16; i += kFThreads) reinterpret_cast<uint4*>(smem + lay.x_off)[i] = src[i];
  }
  __syncthreads();

  // ---- copy warps
  if (warp > kFConsumers) {
    const int nw = min(max(a.fetch_warps, 1), kFCopyWarps);
    if (a.nx.hdr && warp - (kFConsumers + 1) < nw) fused_fetch(a.nx, threadIdx.x - (kFConsumers + 1) * 32, nw);
    return;
  }

  // ---- producer warp
  if (warp == kFConsumers) {
    if (lane == 0) {
      wait_ready_flag(a);  // copy-engine mode: the slots' bytes are in place
      for (int u = 0; u < n_u && c1 > c0; ++u)
        prefetch_l2(a.pool + (long long)p_slot[u] * a.expert_bytes + wd_off + c0 * row_d,
                    (uint32_t)((c1 - c0) * row_d));
      int i = 0;
      bool go = true;
      auto issue = [&](const uint8_t* s0, uint32_t b0, const uint8_t* s1, uint32_t b1) {
        const int s = i % kFStages;
        if (i >= kFStages && !fwait(&empty[s], ((i / kFStages) - 1) & 1, a.status, abort_flag)) {
          go = false;
          return;
        }
        mbar_expect_tx(&full[s], b0 + b1);
        bulk_g2s(ring + (size_t)s * SB, s0, b0, &full[s]);
        if (b1) bulk_g2s(ring + (size_t)s * SB + b0, s1, b1, &full[s]);
        ++i;
      };
      for (int q = q0; q < q1 && go;) {
        const int u = q / I, r = q - u * I;
        const int R = min(min(lay.R, I - r), q1 - q);
        const uint8_t* blob = a.pool + (long long)p_slot[u] * a.expert_bytes;
        issue(blob + r * row_g, (uint32_t)(R * row_g), blob + (I + r) * row_g, (uint32_t)(R * row_g));
        q += R;
      }
      for (int p0 = c0; p0 < c1 && go; p0 += lay.PR) {
        const int PR = min(lay.PR, c1 - p0);
        const int EU = max(1, SB / (int)(PR * row_d));  // experts per unit
        for (int ub = 0; ub < n_u && go; ub += EU) {
          const int s = i % kFStages;
          if (i >= kFStages && !fwait(&empty[s], ((i / kFStages) - 1) & 1, a.status, abort_flag)) {
            go = false;
            break;
          }
          const int ne = min(EU, n_u - ub);
          mbar_expect_tx(&full[s], (uint32_t)(ne * PR * row_d));
          for (int k2 = 0; k2 < ne; ++k2)
            bulk_g2s(ring + (size_t)s * SB + (size_t)k2 * PR * row_d,
                     a.pool + (long long)p_slot[ub + k2] * a.expert_bytes + wd_off + p0 * row_d,
                     (uint32_t)(PR * row_d), &full[s]);
          ++i;
        }
      }
      // no copy may still be writing this CTA's shared memory when it exits
      // (bounded, and not cut short by an abort)
      for (int j = i - kFStages < 0 ? 0 : i - kFStages; j < i; ++j)
        mbar_wait(&full[j % kFStages], (j / kFStages) & 1, a.status);
    }
    return;
  }

  // ---- consumers, phase 1: gate/up + SwiGLU
  const int ctid = threadIdx.x;  // 0 .. 255
  int unit = 0;
  {
    const int sblk = H / 128;
    const int nch = (int)(row_g / 16);  // 16-byte chunks per row
    const int group = warp >> 2, gw = warp & 3;
    for (int q = q0; q < q1; ++unit) {
      const int u = q / I, r = q - u * I;
      const int R = min(min(lay.R, I - r), q1 - q);
      q += R;
      if ((unit & 1) != group) continue;  // the other group's unit
      const int s = unit % kFStages;
      const bool ok = stage_acquire(&full[s], (unit / kFStages) & 1, a.status, abort_flag);
      const int row0 = p_off[u];
      const int nrows = min(p_off[u + 1] - row0, MR);
      const uint8_t* blob = a.pool + (long long)p_slot[u] * a.expert_bytes;
      const uint8_t* xrow[MR];
#pragma unroll
      for (int t = 0; t < MR; ++t)
        xrow[t] = xs + (size_t)(t < nrows ? p_rows[row0 + t] / k : 0) * H * act_bytes;
      for (int jp = gw; jp < R && ok; jp += 4) {
        const uint4* grow = reinterpret_cast<const uint4*>(ring + (size_t)s * SB + jp * row_g);
        const uint4* urow = reinterpret_cast<const uint4*>(ring + (size_t)s * SB + (R + jp) * row_g);
        const int rr = r + jp;
        float ag[MR], au[MR];
#pragma unroll
        for (int t = 0; t < MR; ++t) ag[t] = au[t] = 0.0f;
#pragma unroll
        for (int i = 0; i < NCL; ++i) {
          const int c = i * 32 + lane;
          if (c < nch) {
            float fg[EPC], fu[EPC];
            decode_chunk<WT>(grow[c], fg);
            decode_chunk<WT>(urow[c], fu);
            float sg = 1.0f, su = 1.0f;
            if (WT == FT_W_FP8E4M3_B128) {
              const int cb = (c * EPC) >> 7;
              sg = scale_at(blob, scale_off, (rr >> 7) * sblk + cb);
              su = scale_at(blob, scale_off, (I / 128) * sblk + (rr >> 7) * sblk + cb);
            }
#pragma unroll
            for (int t = 0; t < MR; ++t) {
              if (t < nrows) {
                float xv[EPC];
                load_act<kF32, EPC>(xrow[t], c * EPC, xv);
                float pg0 = 0.0f, pg1 = 0.0f, pu0 = 0.0f, pu1 = 0.0f;
#pragma unroll
                for (int e = 0; e < EPC; e += 2) {
                  pg0 = fmaf(fg[e], xv[e], pg0);
                  pu0 = fmaf(fu[e], xv[e], pu0);
                  pg1 = fmaf(fg[e + 1], xv[e + 1], pg1);
                  pu1 = fmaf(fu[e + 1], xv[e + 1], pu1);
                }
                ag[t] = fmaf(sg, pg0 + pg1, ag[t]);
                au[t] = fmaf(su, pu0 + pu1, au[t]);
              }
            }
          }
        }
#pragma unroll
        for (int t = 0; t < MR; ++t) {
          if (t < nrows) {
            const float g = warp_sum(ag[t]);
            const float v = warp_sum(au[t]);
            if (lane == t) a.h[(long long)p_rows[row0 + t] * I + rr] = g / (1.0f + expf(-g)) * v;
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_n(&empty[s], 2);  // four warps of a group stand for the eight
    }
  }

  // ---- every CTA's h is written and visible after this (bounded)
  __threadfence();
  consumers_sync();
  if (ctid == 0) {
    unsigned* count = a.gbar;
    unsigned* gen = a.gbar + 1;
    const unsigned g = *reinterpret_cast<volatile unsigned*>(gen);
    if (atomicAdd(count, 1u) == gridDim.x - 1) {
      *reinterpret_cast<volatile unsigned*>(count) = 0u;
      __threadfence();
      atomicExch(gen, g + 1u);
    } else {
      const unsigned long long t0 = global_ns();
      while (*reinterpret_cast<volatile unsigned*>(gen) == g) {
        if (global_ns() - t0 > kWaitLimitNs) {
          if (a.status) atomicCAS(a.status, 0, (int)FT_ERR_TIMEOUT);
          *abort_flag = 1;
          break;
        }
      }
    }
    __threadfence();
  }
  consumers_sync();
  const bool h_in_smem = lay.h_bytes > 0;
  if (h_in_smem) {
    const int n4 = rows_total * I / 4;
    const float4* src = reinterpret_cast<const float4*>(a.h);
    for (int i = ctid; i < n4; i += kFConsumers * 32) reinterpret_cast<float4*>(hs)[i] = __ldcg(src + i);
    consumers_sync();
  }
  // ---- consumers, phase 2: down projection + gate-weighted combine
  if (h_in_smem)
    fused_phase2<WT, MR, DCL, true>(a, lay, ring, full, empty, abort_flag, p_slot, p_off, p_rows, p_w, hs, n_u, c0,
                                    c1, unit);
  else
    fused_phase2<WT, MR, DCL, false>(a, lay, ring, full, empty, abort_flag, p_slot, p_off, p_rows, p_w, a.h, n_u,
                                     c0, c1, unit);

  // ---- copy-engine mode: the last CTA to finish tells the copy thread that
  // this event's slots are no longer read (every bulk copy of every CTA has
  // been consumed by now)
  if (a.done_host) {
    consumers_sync();
    if (ctid == 0) {
      __threadfence();
      if (atomicAdd(a.gbar + 2, 1u) == gridDim.x - 1) {
        *reinterpret_cast<volatile unsigned*>(a.gbar + 2) = 0u;
        const int ev = __ldg(&a.hdr[PH_EVENT]);
        __threadfence_system();
        asm volatile("st.release.sys.global.b32 [%0], %1;" ::"l"(a.done_host + (ev % kRing)), "r"(ev) : "memory");
      }
    }
  }
}

__global__ void signal_done_kernel(const int32_t* hdr, int32_t* done_host) {
  const int ev = *reinterpret_cast<const volatile int32_t*>(hdr + PH_EVENT);
  __threadfence_system();
  asm volatile("st.release.sys.global.b32 [%0], %1;" ::"l"(done_host + (ev % kRing)), "r"(ev) : "memory");
}

int num_sms() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
  }
  return n;
}

// CTAs per SM of `kernel` at `smem` bytes of dynamic shared memory (cached
// per size).  The kernel's shared-memory limit only ever grows, to the
// largest size seen: lowering it for a smaller launch would make a later,
// larger launch of the same kernel fail.
template <typename K>
int blocks_per_sm_t(K kernel, int threads, int smem, cudaError_t* err) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> cache;
  static std::map<const void*, int> limit;
  std::lock_guard<std::mutex> lk(mu);
  const auto key = std::make_pair(reinterpret_cast<const void*>(kernel), smem * 4096 + threads);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  int& lim = limit[reinterpret_cast<const void*>(kernel)];
  if (smem > lim) {
    *err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (*err == cudaSuccess)  // same split as the route and fetch kernels, so they can share an SM
      *err = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                  cudaSharedmemCarveoutMaxShared);
    if (*err != cudaSuccess) return 0;
    lim = smem;
  }
  int per_sm = 1;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem);
  if (per_sm < 0) per_sm = 0;
  cache[key] = per_sm;
  return per_sm;
}

template <typename K>
int blocks_per_sm(K kernel, int smem, cudaError_t* err) {
  const int n = blocks_per_sm_t(kernel, kThreads, smem, err);
  return n < 1 ? 1 : n;
}

template <int WT>
cudaError_t gateup_typed(const FfnArgs& a, cudaStream_t s) {
  const GateUpLayout lay(a.H, a.I, a.T, W<WT>::kBytes, WT == FT_W_F32 ? 4 : 2, a.max_unique, a.T * a.k);
  cudaError_t e = cudaSuccess;
  const int per_sm = blocks_per_sm(gateup_kernel<WT>, lay.total, &e);
  if (e != cudaSuccess) return e;
  // units = n_u * I / P is only known on the device; the grid covers the
  // largest batch (max_unique experts) within one wave
  const int max_units = a.max_unique * (a.I / lay.P);
  int grid = num_sms() * per_sm;
  if (grid > max_units) grid = max_units;
  if (grid < 1) grid = 1;
  gateup_kernel<WT><<<grid, kThreads, lay.total, s>>>(a);
  return cudaGetLastError();
}

template <int WT>
cudaError_t down_typed(const FfnArgs& a, cudaStream_t s) {
  const DownLayout lay(a.I, W<WT>::kBytes, a.max_unique, a.T * a.k);
  cudaError_t e = cudaSuccess;
  const int per_sm = blocks_per_sm(down_kernel<WT>, lay.total, &e);
  if (e != cudaSuccess) return e;
  const int n_rb = a.H / lay.RD;
  int grid = num_sms() * per_sm;
  if (grid > n_rb) grid = n_rb;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = lay.total;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, down_kernel<WT>, a);
}

template <int WT, int MR, int NCL, int DCL>
cudaError_t fused_launch(const FfnArgs& a, const FusedLayout& lay, int grid, cudaStream_t s) {
  cudaError_t e = cudaSuccess;
  const int per_sm = blocks_per_sm_t(ffn_fused_kernel<WT, MR, NCL, DCL>, kFThreads, lay.total, &e);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorNotSupported;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kFThreads);
  cfg.dynamicSmemBytes = lay.total;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {const_cast<FfnArgs*>(&a)};
  return cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(ffn_fused_kernel<WT, MR, NCL, DCL>), args);
}

template <int WT>
cudaError_t fused_typed(const FfnArgs& a, cudaStream_t s) {
  const int grid = num_sms();  // one CTA per SM, all co-resident
  const FusedLayout lay(a.H, a.I, a.T, W<WT>::kBytes, WT == FT_W_F32 ? 4 : 2, a.max_unique, a.T * a.k);
  if (!lay.ok() || lay.total > kFusedSmemBudget + 1024 || !a.gbar || a.T > kMaxRows) return cudaErrorNotSupported;
  // One row shape per weight type has an instantiation (16-byte chunks per
  // lane of a Wg/Wu row, of a Wd row): fp32 H 256 / I 128 (1 KB, 512 B),
  // bf16 H 2048 / I 512 (4 KB, 1 KB), fp8 H 4096 / I 2048 (4 KB, 2 KB).
  // Other shapes take the two-kernel path.
  constexpr int NCL = WT == FT_W_F32 ? 2 : 8;
  constexpr int DCL = WT == FT_W_F32 ? 1 : (WT == FT_W_BF16 ? 2 : 4);
  const int nch = a.H * W<WT>::kBytes / 16, dch = a.I * W<WT>::kBytes / 16;
  if (nch > 32 * NCL || nch <= 32 * NCL - 64 || dch != 32 * DCL) return cudaErrorNotSupported;
  return a.T == 1 ? fused_launch<WT, 1, NCL, DCL>(a, lay, grid, s) : fused_launch<WT, kMaxRows, NCL, DCL>(a, lay, grid, s);
}

}  // namespace

cudaError_t launch_signal_done(const FfnArgs& a, cudaStream_t s) {
  signal_done_kernel<<<1, 1, 0, s>>>(a.hdr, a.done_host);
  return cudaGetLastError();
}

cudaError_t launch_decode_ffn_fused(const FfnArgs& a, cudaStream_t s) {
  switch (a.wdtype) {
    case FT_W_F32: return fused_typed<FT_W_F32>(a, s);
    case FT_W_BF16: return fused_typed<FT_W_BF16>(a, s);
    case FT_W_FP8E4M3_B128: return fused_typed<FT_W_FP8E4M3_B128>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_gateup(const FfnArgs& a, cudaStream_t s) {
  switch (a.wdtype) {
    case FT_W_F32: return gateup_typed<FT_W_F32>(a, s);
    case FT_W_BF16: return gateup_typed<FT_W_BF16>(a, s);
    case FT_W_FP8E4M3_B128: return gateup_typed<FT_W_FP8E4M3_B128>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_down(const FfnArgs& a, cudaStream_t s) {
  if (a.H % kConsumerWarps) return cudaErrorInvalidValue;
  switch (a.wdtype) {
    case FT_W_F32: return down_typed<FT_W_F32>(a, s);
    case FT_W_BF16: return down_typed<FT_W_BF16>(a, s);
    case FT_W_FP8E4M3_B128: return down_typed<FT_W_FP8E4M3_B128>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ft
