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

__device__ __forceinline__ uint4 ldg16(const uint4* p) { return __ldg(p); }

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
// One CTA per SM, all co-resident (cooperative launch), 12 warps.
//  prologue: thread 0 bulk-copies this CTA's Wd rows (a contiguous range of
//            output columns, one copy per expert, as many experts as fit) into
//            shared memory; they do not depend on h, so they stream during
//            phase 1;
//  phase 1:  one warp per (expert, intermediate row) task: the Wg and Wu rows
//            are read with 16-byte loads, all issued before the arithmetic;
//            the warp writes h = silu(g) * u for each token of the expert;
//  barrier:  grid-wide (bounded), h complete everywhere;
//  phase 2:  one warp per output column of the CTA's range: sum over experts
//            (ascending) and their rows of w * (Wd row . h row).
// The CTA stays small (384 threads, <= 96 registers, <= 150 KB shared
// memory) so that a route CTA and a fetch CTA can run on the same SM.
constexpr int kFThreads = 384;
constexpr int kFWarps = kFThreads / 32;
constexpr int kFusedSmemBudget = 150 * 1024;

struct FusedLayout {
  int cols_max, x_off, h_off, h_bytes, plan_off, w_off, wd_off, wd_cap, bar_off, total;
  __host__ __device__ FusedLayout(int H, int I, int T, int wsize, int act_bytes, int max_unique, int rows,
                                  int grid) {
    cols_max = (H + grid - 1) / grid;  // output columns per CTA
    x_off = 0;
    h_off = align_up(T * H * act_bytes, 16);
    h_bytes = rows * I * 4;
    if (h_bytes > 32 * 1024) h_bytes = 0;  // larger h is read from L2
    plan_off = align_up(h_off + h_bytes, 16);
    w_off = plan_off + plan_bytes(max_unique, rows);
    wd_off = align_up(w_off + rows * 4, 128);
    const int per_expert = align_up(cols_max * I * wsize, 128);
    wd_cap = (kFusedSmemBudget - wd_off - 64) / per_expert;  // experts whose Wd rows fit
    if (wd_cap < 0) wd_cap = 0;
    if (wd_cap > max_unique) wd_cap = max_unique;
    bar_off = wd_off + wd_cap * per_expert;
    total = bar_off + 16;
  }
};

// NC: 16-byte chunks per lane per gate/up row (H*wsize <= 512*NC); MR: most
// rows (tokens) of one expert, 1 for single-token decode.
template <int WT, int NC, int MR>
__global__ void __maxnreg__(96) ffn_fused_kernel(FfnArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr bool kF32 = WT == FT_W_F32;
  constexpr int EPC = W<WT>::kEPC, WSZ = W<WT>::kBytes;
  const int H = a.H, I = a.I, k = a.k, T = a.T;
  const int act_bytes = kF32 ? 4 : 2;
  const int rows_total = T * k;
  const FusedLayout lay(H, I, T, WSZ, act_bytes, a.max_unique, rows_total, gridDim.x);
  uint8_t* xs = smem + lay.x_off;
  float* hs = reinterpret_cast<float*>(smem + lay.h_off);
  int32_t* p_slot = reinterpret_cast<int32_t*>(smem + lay.plan_off);
  int32_t* p_off = p_slot + a.max_unique;
  int32_t* p_rows = p_off + a.max_unique + 1;
  float* p_w = reinterpret_cast<float*>(smem + lay.w_off);
  uint8_t* wds = smem + lay.wd_off;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + lay.bar_off);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_u = min(__ldg(&a.hdr[PH_UNIQUE]), a.max_unique);
  // this CTA's output columns [c0, c1), balanced and contiguous
  const int c0 = (int)((long long)H * blockIdx.x / gridDim.x);
  const int c1 = (int)((long long)H * (blockIdx.x + 1) / gridDim.x);
  const long long d_row_bytes = (long long)I * WSZ;
  const int per_expert = align_up(lay.cols_max * I * WSZ, 128);
  const long long wd_off = 2LL * H * I * WSZ;
  const int n_pref = min(n_u, lay.wd_cap);  // experts whose Wd rows are in shared memory

  if (threadIdx.x == 0) {
    wait_ready_flag(a);
    mbar_init(bar, 1);
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
    for (int i = threadIdx.x; i < n16; i += kFThreads) reinterpret_cast<uint4*>(xs)[i] = src[i];
  }
  __syncthreads();
  if (threadIdx.x == 0 && n_pref > 0 && c1 > c0) {
    const uint32_t bytes = (uint32_t)((c1 - c0) * d_row_bytes);
    mbar_expect_tx(bar, bytes * n_pref);
    for (int u = 0; u < n_pref; ++u)
      bulk_g2s(wds + (size_t)u * per_expert,
               a.pool + (long long)p_slot[u] * a.expert_bytes + wd_off + (long long)c0 * d_row_bytes, bytes, bar);
  }

  // ---- phase 1: gate/up
  const long long g_row_bytes = (long long)H * WSZ;
  const long long scale_off = 3LL * H * I * WSZ;
  const int nch = H / EPC;
  {
    const int sblk = H / 128;
    const int gw = blockIdx.x * kFWarps + warp, nw = gridDim.x * kFWarps;
    for (int task = gw; task < n_u * I; task += nw) {
      const int u = task / I, r = task - u * I;
      const uint8_t* blob = a.pool + (long long)p_slot[u] * a.expert_bytes;
      const uint4* grow = reinterpret_cast<const uint4*>(blob + (long long)r * g_row_bytes);
      const uint4* urow = reinterpret_cast<const uint4*>(blob + (long long)(I + r) * g_row_bytes);
      uint4 wg[NC], wu[NC];
#pragma unroll
      for (int i = 0; i < NC; ++i) {
        const int c = i * 32 + lane;
        if (c < nch) {
          wg[i] = ldg16(grow + c);
          wu[i] = ldg16(urow + c);
        }
      }
      const int row0 = p_off[u];
      const int nrows = min(p_off[u + 1] - row0, MR);
      float ag[MR], au[MR];
#pragma unroll
      for (int q = 0; q < MR; ++q) ag[q] = au[q] = 0.0f;
#pragma unroll
      for (int i = 0; i < NC; ++i) {
        const int c = i * 32 + lane;
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
          for (int q = 0; q < MR; ++q) {
            if (q < nrows) {
              float xv[EPC];
              load_act<kF32, EPC>(xs + (size_t)(p_rows[row0 + q] / k) * H * act_bytes, c * EPC, xv);
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
#pragma unroll
      for (int q = 0; q < MR; ++q) {
        if (q < nrows) {
          const float g = warp_sum(ag[q]);
          const float v = warp_sum(au[q]);
          if (lane == 0) a.h[(long long)p_rows[row0 + q] * I + r] = g / (1.0f + expf(-g)) * v;
        }
      }
    }
  }

  // ---- every CTA's h is written and visible after this (bounded)
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned* count = a.gbar;
    unsigned* gen = a.gbar + 1;
    __threadfence();
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
          break;
        }
      }
    }
    __threadfence();
  }
  __syncthreads();

  // ---- phase 2: down + combine
  const bool h_in_smem = lay.h_bytes > 0;
  if (h_in_smem) {
    const int n4 = rows_total * I / 4;
    const float4* src = reinterpret_cast<const float4*>(a.h);
    for (int i = threadIdx.x; i < n4; i += kFThreads) reinterpret_cast<float4*>(hs)[i] = __ldcg(src + i);
    __syncthreads();
  }
  const float* hbase = h_in_smem ? hs : a.h;
  bool wd_ready = true;
  if (n_pref > 0 && c1 > c0) {  // every thread acquires the bulk copies' completion
    if (lane == 0) wd_ready = mbar_wait(bar, 0, a.status);
    wd_ready = __shfl_sync(0xffffffffu, wd_ready, 0);
    if (wd_ready) mbar_try_wait(bar, 0);
  }
  const int dch = I / EPC;
  const int sblk = I / 128;
  const int sbase = 2 * (I / 128) * (H / 128);
  for (int cc = c0 + warp; cc < c1; cc += kFWarps) {
    float acc[MR];
#pragma unroll
    for (int q = 0; q < MR; ++q) acc[q] = 0.0f;
    for (int u = 0; u < n_u; ++u) {
      const uint8_t* blob = a.pool + (long long)p_slot[u] * a.expert_bytes;
      const uint4* wrow = (u < n_pref && wd_ready)
                              ? reinterpret_cast<const uint4*>(wds + (size_t)u * per_expert + (cc - c0) * d_row_bytes)
                              : reinterpret_cast<const uint4*>(blob + wd_off + (long long)cc * d_row_bytes);
      const int row0 = p_off[u];
      const int nrows = min(p_off[u + 1] - row0, MR);
      float part[MR];
#pragma unroll
      for (int q = 0; q < MR; ++q) part[q] = 0.0f;
      for (int c = lane; c < dch; c += 32) {
        float f[EPC];
        decode_chunk<WT>(u < n_pref && wd_ready ? wrow[c] : ldg16(wrow + c), f);
        float sc = 1.0f;
        if (WT == FT_W_FP8E4M3_B128) sc = scale_at(blob, scale_off, sbase + (cc >> 7) * sblk + ((c * EPC) >> 7));
#pragma unroll
        for (int q = 0; q < MR; ++q) {
          if (q < nrows) {
            const float4* hp = reinterpret_cast<const float4*>(hbase + (long long)p_rows[row0 + q] * I + c * EPC);
            float p = 0.0f;
#pragma unroll
            for (int e4 = 0; e4 < EPC / 4; ++e4) {
              const float4 hv = h_in_smem ? hp[e4] : __ldcg(hp + e4);
              p = fmaf(f[4 * e4], hv.x, p);
              p = fmaf(f[4 * e4 + 1], hv.y, p);
              p = fmaf(f[4 * e4 + 2], hv.z, p);
              p = fmaf(f[4 * e4 + 3], hv.w, p);
            }
            part[q] = fmaf(sc, p, part[q]);
          }
        }
      }
#pragma unroll
      for (int q = 0; q < MR; ++q) {
        if (q < nrows) {
          const int row = p_rows[row0 + q];
          const int t = row / k;
#pragma unroll
          for (int tt = 0; tt < MR; ++tt)
            if (tt == t) acc[tt] = fmaf(p_w[row], part[q], acc[tt]);
        }
      }
    }
#pragma unroll
    for (int t = 0; t < MR; ++t) {
      if (t < T) {
        const float v = warp_sum(acc[t]);
        if (lane == 0) a.y[(long long)t * H + cc] = v;
      }
    }
  }
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

// CTAs per SM of `kernel` at `smem` bytes of dynamic shared memory; sets the
// kernel's shared-memory limit the first time a size is seen (cached).
template <typename K>
int blocks_per_sm_t(K kernel, int threads, int smem, cudaError_t* err) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> cache;
  std::lock_guard<std::mutex> lk(mu);
  const auto key = std::make_pair(reinterpret_cast<const void*>(kernel), smem * 4096 + threads);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  *err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (*err != cudaSuccess) return 0;
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

template <int WT>
cudaError_t fused_typed(const FfnArgs& a, cudaStream_t s) {
  constexpr int EPC = W<WT>::kEPC;
  const int nch = a.H / EPC;
  const int grid = num_sms();  // one CTA per SM, all co-resident
  const FusedLayout lay(a.H, a.I, a.T, W<WT>::kBytes, WT == FT_W_F32 ? 4 : 2, a.max_unique, a.T * a.k, grid);
  if (lay.total > kFusedSmemBudget + 1024 || !a.gbar || nch > 32 * 8) return cudaErrorNotSupported;
  const void* fn;
  cudaError_t e = cudaSuccess;
  int per_sm = 0;
  if (a.T == 1) {
    fn = nch <= 64 ? reinterpret_cast<const void*>(ffn_fused_kernel<WT, 2, 1>)
                   : reinterpret_cast<const void*>(ffn_fused_kernel<WT, 8, 1>);
    per_sm = nch <= 64 ? blocks_per_sm_t(ffn_fused_kernel<WT, 2, 1>, kFThreads, lay.total, &e)
                       : blocks_per_sm_t(ffn_fused_kernel<WT, 8, 1>, kFThreads, lay.total, &e);
  } else {
    fn = nch <= 64 ? reinterpret_cast<const void*>(ffn_fused_kernel<WT, 2, kMaxRows>)
                   : reinterpret_cast<const void*>(ffn_fused_kernel<WT, 8, kMaxRows>);
    per_sm = nch <= 64 ? blocks_per_sm_t(ffn_fused_kernel<WT, 2, kMaxRows>, kFThreads, lay.total, &e)
                       : blocks_per_sm_t(ffn_fused_kernel<WT, 8, kMaxRows>, kFThreads, lay.total, &e);
  }
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
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace

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
