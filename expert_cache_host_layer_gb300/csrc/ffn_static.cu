// ft_moe_decode_ffn_static: the decode expert FFN for callers that cannot
// allocate device memory.
//
// Some callers may not call cudaMalloc at all: an engine whose memory planner
// hands out every byte of device memory up front and forbids allocation
// afterwards, or a latency-critical serving loop where cudaMalloc/cudaFree
// would stall (cudaFree synchronises the whole device).  ft_moe_forward needs
// a cache handle, and ft_cache_create allocates its tables and buffers; this
// entry point needs neither.  Its working memory (the per-call expert
// grouping and the fp32 intermediate h) lives in one file-scope __device__
// array.  With lazy module loading (the CUDA default) the array is reserved
// on a GPU when the library's module is first loaded there - at the first
// call on that device - and kept until the process exits; with
// CUDA_MODULE_LOADING=EAGER it is reserved when the library loads.
//
// The array is shared by all calls on a device and keeps whatever the last
// call left in it.  Each call first rewrites every plan word it later reads,
// so nothing there has to start at zero; the status word is the exception: it
// starts at zero (static storage), a bounded wait that runs out sets it, and
// only ft_moe_decode_ffn_static_status reads and clears it.  Two calls whose
// kernels overlap on the GPU (different streams, or different host threads)
// race on the array and produce garbage.  Serialise them on one stream.
#include <algorithm>
#include <climits>
#include <mutex>
#include <string>

#include "driver_api.h"
#include "ft_internal.h"

namespace ft {
namespace {

constexpr size_t kScratchBytes = size_t(1) << 20;   // 1 MiB
constexpr int kStatusWords = 16;                      // word 0: sticky status of the kernels' bounded waits
constexpr int kPlanWords = 4096;                      // status, header, unique_slot, u_offset, rows_by_u
constexpr size_t kHBytes = kScratchBytes - kPlanWords * sizeof(int32_t);

static __device__ __align__(256) unsigned char g_ffn_scratch[kScratchBytes];

// Device address of g_ffn_scratch per device ordinal, with the context it was
// looked up in: a different current context (after cudaDeviceReset, or a
// context the caller created) gets the address looked up again.
struct ScratchAddr {
  CUcontext ctx = nullptr;
  void* addr = nullptr;
};
std::mutex g_mu;
ScratchAddr g_scratch_addr[64];

ft_status scratch_base(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
    return set_error(FT_ERR_CUDA, "cudaGetDevice failed or device ordinal >= 64");
  const CUcontext ctx = current_context();
  std::lock_guard<std::mutex> lk(g_mu);
  ScratchAddr& a = g_scratch_addr[dev];
  if (!a.addr || a.ctx != ctx) {  // first call on this device (or in this context): look the address up
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_ffn_scratch);
    if (e != cudaSuccess || !p)
      return set_error(FT_ERR_CUDA, "cudaGetSymbolAddress of the static scratch: %s", cudaGetErrorString(e));
    a.addr = p;
    a.ctx = ctx;
  }
  *out = a.addr;
  return FT_OK;
}

// Groups the T*k (token, pick) rows by expert: the plan the decode FFN kernels read.
__global__ void static_plan_kernel(const int32_t* topk_idx, int T, int k, int E, const int32_t* expert_slot,
                                   long long num_slots, int32_t* hdr, int32_t* unique_slot, int32_t* u_offset,
                                   int32_t* rows_by_u) {
  __shared__ uint32_t s_bits[kMaxExperts / 32];
  __shared__ int s_pre[33];
  __shared__ int s_row_u[kDecodeMaxTokens * kMaxTopK];
  __shared__ int s_cnt[kMaxExperts];
  __shared__ int s_uexp[kMaxExperts];
  const int tid = threadIdx.x, rows = T * k, nwords = (E + 31) >> 5;
  for (int i = tid; i < nwords; i += blockDim.x) s_bits[i] = 0u;
  for (int i = tid; i < E; i += blockDim.x) s_cnt[i] = 0;
  __syncthreads();
  // valid picks: expert id in range and held by a slot in range
  for (int r = tid; r < rows; r += blockDim.x) {
    const int e = topk_idx[r];
    const bool ok = e >= 0 && e < E && expert_slot[e] >= 0 && expert_slot[e] < num_slots;
    s_row_u[r] = ok ? e : -1;
    if (ok) {
      atomicOr(&s_bits[e >> 5], 1u << (e & 31));
      atomicAdd(&s_cnt[e], 1);
    }
  }
  __syncthreads();
  if (tid < 32) {
    int c = tid < nwords ? __popc(s_bits[tid]) : 0;
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, c, o);
      if (tid >= o) c += y;
    }
    s_pre[tid + 1] = c;
    if (tid == 0) s_pre[0] = 0;
  }
  __syncthreads();
  const int n_u = s_pre[nwords];
  for (int e = tid; e < E; e += blockDim.x) {
    const int w = e >> 5, b = e & 31;
    if ((s_bits[w] >> b) & 1u) s_uexp[s_pre[w] + __popc(s_bits[w] & ((1u << b) - 1u))] = e;
  }
  __syncthreads();
  if (tid == 0) {  // offsets in ascending expert order (n_u <= T*k is small)
    int off = 0;
    for (int u = 0; u < n_u; ++u) {
      u_offset[u] = off;
      unique_slot[u] = expert_slot[s_uexp[u]];
      off += s_cnt[s_uexp[u]];
    }
    u_offset[n_u] = off;
    for (int i = 0; i < PH_WORDS; ++i) hdr[i] = 0;
    hdr[PH_TOKENS] = T;
    hdr[PH_UNIQUE] = n_u;
    hdr[PH_ROWS] = rows;
  }
  __syncthreads();
  for (int r = tid; r < rows; r += blockDim.x) {
    const int e = s_row_u[r];
    if (e < 0) continue;
    int u = 0;
    while (s_uexp[u] != e) ++u;  // n_u <= rows <= 256
    int before = 0;
    for (int q = 0; q < r; ++q) before += s_row_u[q] == e;
    rows_by_u[u_offset[u] + before] = r;
  }
}

}  // namespace
}  // namespace ft

using namespace ft;

extern "C" ft_status ft_moe_decode_ffn_static(int32_t hidden, int32_t inter, int32_t wdtype, int32_t num_experts,
                                              int32_t top_k, const void* slot_pool, int64_t num_slots,
                                              const int32_t* expert_slot, const int32_t* topk_idx,
                                              const float* topk_w, const void* x, int32_t T, void* y,
                                              void* stream) {
  const size_t eb = ft_expert_bytes(hidden, inter, wdtype);
  if (eb == 0 || (wdtype != FT_W_F32 && (hidden % 128 || inter % 128)))
    return set_error(FT_ERR_INVALID_ARG, "unsupported hidden/inter/wdtype (%d, %d, %d)", hidden, inter, wdtype);
  if (hidden % 8)  // the down kernel gives each of its 8 consumer warps one output column per block of 8
    return set_error(FT_ERR_INVALID_ARG, "hidden=%d is not a multiple of 8", hidden);
  if (num_experts < 1 || num_experts > kMaxExperts || top_k < 1 || top_k > kMaxTopK || top_k > num_experts)
    return set_error(FT_ERR_INVALID_ARG, "num_experts must be 1..%d and top_k 1..min(num_experts, %d)", kMaxExperts,
                     kMaxTopK);
  if (T < 0 || T > kDecodeMaxTokens)
    return set_error(FT_ERR_INVALID_ARG, "T=%d outside 0..%d (decode batches only)", T, kDecodeMaxTokens);
  if (T == 0) return FT_OK;
  if (!slot_pool || num_slots < 1 || !expert_slot || !topk_idx || !topk_w || !x || !y)
    return set_error(FT_ERR_INVALID_ARG, "null pointer or num_slots < 1");
  // the scratch limit: status + header + unique_slot[E] + u_offset[E+1] + rows in the plan area, T*k*I floats for h
  const long long rows = (long long)T * top_k;
  const long long plan_words = kStatusWords + PH_WORDS + 2LL * num_experts + 1 + rows;
  if (plan_words > kPlanWords)
    return set_error(FT_ERR_INVALID_ARG, "plan of %lld words exceeds the static scratch plan area of %d words",
                     plan_words, kPlanWords);
  if ((size_t)rows * inter * sizeof(float) > kHBytes)
    return set_error(FT_ERR_INVALID_ARG,
                     "T*top_k*inter*4 = %lld bytes exceeds the %zu-byte static scratch for the intermediate h",
                     rows * inter * 4LL, kHBytes);

  void* base = nullptr;
  const ft_status st = scratch_base(&base);
  if (st != FT_OK) return st;
  int32_t* w = static_cast<int32_t*>(base);
  int32_t* status = w;
  int32_t* hdr = w + kStatusWords;
  int32_t* unique_slot = hdr + PH_WORDS;
  int32_t* u_offset = unique_slot + num_experts;
  int32_t* rows_by_u = u_offset + num_experts + 1;
  float* h = reinterpret_cast<float*>(static_cast<unsigned char*>(base) + kPlanWords * sizeof(int32_t));

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  static_plan_kernel<<<1, 256, 0, s>>>(topk_idx, T, top_k, num_experts, expert_slot, num_slots, hdr, unique_slot,
                                       u_offset, rows_by_u);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(FT_ERR_CUDA, "plan kernel launch: %s", cudaGetErrorString(e));
  FfnArgs f{};
  f.hdr = hdr; f.unique_slot = unique_slot; f.u_offset = u_offset; f.rows_by_u = rows_by_u; f.topk_w = topk_w;
  f.x = x; f.y = static_cast<float*>(y); f.pool = static_cast<const uint8_t*>(slot_pool);
  f.expert_bytes = (long long)eb; f.num_slots = (int)std::min<long long>(num_slots, INT_MAX);
  f.H = hidden; f.I = inter; f.k = top_k; f.T = T; f.wdtype = wdtype; f.h = h;
  f.max_unique = (int)std::min<long long>(rows, num_experts);
  f.status = status;
  if ((e = launch_decode_gateup(f, s)) != cudaSuccess)
    return set_error(FT_ERR_CUDA, "gate/up launch: %s", cudaGetErrorString(e));
  if ((e = launch_decode_down(f, s)) != cudaSuccess)
    return set_error(FT_ERR_CUDA, "down launch: %s", cudaGetErrorString(e));
  return FT_OK;
}

extern "C" ft_status ft_moe_decode_ffn_static_status(void* stream) {
  void* base = nullptr;
  ft_status st = scratch_base(&base);
  if (st != FT_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return set_error(FT_ERR_CUDA, "stream synchronize: %s", cudaGetErrorString(e));
  int32_t word = 0;
  e = cudaMemcpy(&word, base, sizeof word, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return set_error(FT_ERR_CUDA, "reading the static status word: %s", cudaGetErrorString(e));
  if (word == FT_OK) return FT_OK;
  const int32_t zero = 0;
  e = cudaMemcpy(base, &zero, sizeof zero, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return set_error(FT_ERR_CUDA, "clearing the static status word: %s", cudaGetErrorString(e));
  return set_error((ft_status)word, "a static-scratch FFN call raised %s", ft_status_str((ft_status)word));
}
