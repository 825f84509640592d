// Decode-path expert FFN (T <= 8 tokens), two-kernel form: two HBM-bound
// kernels that stream the expert weights straight from their cache slots
// through shared memory.  The cache path runs the one-pass fused kernel of
// decode_fused.cu and falls back to these two for shapes that kernel does not
// take; the static-scratch entry point always uses them.
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

#include "decode_common.h"
#include "ft_internal.h"

namespace ft {
namespace {
using namespace dec;

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;  // + one producer warp
constexpr int kMaxRows = kDecodeMaxTokens;           // rows of one expert in a decode batch
__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory"); }
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

// Copies the plan arrays the FFN kernels index into shared memory; in checked
// builds, nonzero if one of this thread's entries is out of range.
__device__ __forceinline__ int stage_plan(const FfnArgs& a, int n_u, int32_t* s_slot, int32_t* s_off,
                                          int32_t* s_rows) {
  const int rows = a.T * a.k;
  int bad = 0;
  for (int i = threadIdx.x; i < n_u; i += blockDim.x) {
    s_slot[i] = __ldg(&a.unique_slot[i]);
    if (kChecked) bad |= s_slot[i] < 0 || s_slot[i] >= a.num_slots;
  }
  for (int i = threadIdx.x; i <= n_u; i += blockDim.x) {
    s_off[i] = __ldg(&a.u_offset[i]);
    if (kChecked) bad |= s_off[i] < 0 || s_off[i] > rows;
  }
  for (int i = threadIdx.x; i < rows; i += blockDim.x) {
    s_rows[i] = __ldg(&a.rows_by_u[i]);
    if (kChecked) bad |= s_rows[i] < 0 || s_rows[i] >= rows;
  }
  return bad;
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
  const bool plan_ok = plan_sync(stage_plan(a, n_u, p_slot, p_off, p_rows), a.status);
  pdl_launch_dependents();  // the down kernel may start streaming Wd now

  const int units_per_u = I / P;
  const int n_units = plan_ok ? n_u * units_per_u : 0;
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
  const int n_u_plan = min(__ldg(&a.hdr[PH_UNIQUE]), a.max_unique);
  if (threadIdx.x == 0) {
    wait_ready_flag(a);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    mbar_init_fence();
  }
  const int n_u = plan_sync(stage_plan(a, n_u_plan, p_slot, p_off, p_rows), a.status) ? n_u_plan : 0;
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

}  // namespace

cudaError_t launch_signal_done(const FfnArgs& a, cudaStream_t s) {
  signal_done_kernel<<<1, 1, 0, s>>>(a.hdr, a.done_host);
  return cudaGetLastError();
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
