// Miss fetch by SM pull: a kernel on the copy stream reads the layer's miss
// list from its device plan and copies each missed expert blob from the host
// bank (mapped pinned memory, read over the host link) into its victim slot.
// No host round trip is needed, so the copy of layer l+1 can be enqueued while
// layer l computes ("FreeToken: az VRAM ile büyük MoE modelleri", intro:
// misses streamed from host RAM; "FreeToken: Efficient Edge-Native MoE Serving
// ...", ablation paragraph: double buffering of the expert transfers).
//
// Work items are 32 KB chunks of the n_miss blobs; each CTA copies one chunk
// per round with 8 independent 16-byte loads in flight per thread (256
// threads: a small CTA that fits beside an FFN CTA on the same SM).
#include "ft_internal.h"

namespace ft {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 8;
constexpr long long kChunk16 = (long long)kThreads * kUnroll;  // 16-byte words per chunk (32 KB)

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.cs.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

__global__ void __launch_bounds__(kThreads) pull_misses_kernel(PullArgs a) {
  int n_miss = __ldcg(&a.hdr[PH_MISS]);
  if (!checked_ok(n_miss >= 0 && n_miss <= a.E, a.status)) n_miss = 0;
  const long long eb16 = a.expert_bytes >> 4;
  const long long chunks_per_blob = (eb16 + kChunk16 - 1) / kChunk16;
  const long long items = (long long)n_miss * chunks_per_blob;
  const uint4* bank = static_cast<const uint4*>(a.bank);
  uint4* pool = static_cast<uint4*>(a.pool);
  for (long long it = blockIdx.x; it < items; it += gridDim.x) {
    const int m = (int)(it / chunks_per_blob);
    const long long c = it - (long long)m * chunks_per_blob;
    const int e = __ldcg(&a.miss_expert[m]);
    const int slot = __ldcg(&a.miss_slot[m]);
    if (!checked_ok(slot >= 0 && slot < a.num_slots && e >= 0 && e < a.E, a.status)) continue;
    const long long blob = ((long long)a.layer * a.E + e) % a.bank_blobs;
    const uint4* src = bank + blob * eb16 + c * kChunk16;
    uint4* dst = pool + (long long)slot * eb16 + c * kChunk16;
    const long long n = min(kChunk16, eb16 - c * kChunk16);
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const long long i = (long long)u * kThreads + threadIdx.x;
      if (i < n) v[u] = ld_stream(src + i);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const long long i = (long long)u * kThreads + threadIdx.x;
      if (i < n) dst[i] = v[u];
    }
  }
}

}  // namespace

cudaError_t prefer_max_shared_fetch() {
  return cudaFuncSetAttribute(pull_misses_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                              cudaSharedmemCarveoutMaxShared);
}

cudaError_t launch_pull_misses(const PullArgs& a, int ctas, cudaStream_t s) {
  pull_misses_kernel<<<ctas, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace ft
