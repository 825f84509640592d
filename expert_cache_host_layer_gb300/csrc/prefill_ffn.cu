// Prefill-path expert FFN (T > 8 tokens per layer event), bf16 weights: the
// token permutation and the two grouped GEMMs of the routed SwiGLU experts,
// reading the weights straight from their cache slots.
//
//   group_rows:  the T*k (token, pick) rows sorted by unique expert (ascending
//                row within an expert): rows_by_u, and pos[row] = its place
//   gate/up:     h[p][i] = silu(Wg[i] . x_t) * (Wu[i] . x_t)  (bf16 h; p the
//                grouped place of row (t, j))
//   down:        yp[p][c] = w_tj * (Wd[c] . h[p])              (fp32)
//   combine:     y[t][c] = sum over j < k, ascending, of yp[pos[t*k+j]][c]
//
// The GEMMs are grouped by expert: a tile is 128 grouped rows of one expert
// by a block of output columns; a persistent grid walks the tiles.  Operands
// move global -> shared with cp.async (16-byte, 3 stages; x rows are gathered
// by token index, rows past the expert's last are zero-filled), fragments come
// from ldmatrix, and mma.sync m16n8k16 bf16 accumulates in fp32.  The gate/up
// tile pairs 64 Wg rows with the same 64 Wu rows so SwiGLU happens in the
// epilogue.  The combine sums each token's picks in a fixed order: the result
// does not depend on how tiles were scheduled.
//
// The grouped SwiGLU expert and its gate-weighted combine follow the routed
// experts of the MoE layers the pages serve ("FreeToken vs vLLM on one RTX
// 3090", "Why the performance differs"; the prefill chunk of "FreeToken:
// Efficient Edge-Native MoE Serving ...", ablation paragraph).
#include <cuda_bf16.h>

#include <mutex>
#include <set>

#include "ft_internal.h"

namespace ft {
namespace {

constexpr int kPThreads = 256;
constexpr int kBM = 128;                 // grouped rows per tile
constexpr int kBK = 32;                  // k per stage
constexpr int kPitch = kBK + 8;          // bf16 per shared row: 80 B keeps ldmatrix conflict-free
constexpr int kStages = 3;
constexpr int kBN1 = 64;                 // gate/up: h columns per tile (64 Wg + 64 Wu rows)
constexpr int kBN2 = 128;                // down: output columns per tile
constexpr int kTileElems = kBM * kPitch;  // one operand tile of 128 rows
constexpr int kHdrInts = 3 * (kMaxExperts + 1);
constexpr int kHdrBytes = (kHdrInts * 4 + 127) / 128 * 128;
constexpr int kGemmSmem = kHdrBytes + kStages * 2 * kTileElems * 2;  // A and B tiles, bf16

__device__ __forceinline__ uint32_t saddr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// 16-byte async copy global -> shared; `valid` false zero-fills (no read).
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(saddr(dst)), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t* r, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(saddr(p)));
}
// c += a (16x16, row) * b (16x8, col), bf16 in, fp32 accumulate
__device__ __forceinline__ void mma_bf16(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Per-CTA tile table: s_off = u_offset, s_pre[u] = m-tiles of the experts
// before u, s_slot = slot of each unique expert.  Returns the m-tile total.
__device__ int tile_table(const PrefillArgs& a, int n_u, int* s_off, int* s_pre, int* s_slot) {
  for (int u = threadIdx.x; u <= n_u; u += kPThreads) s_off[u] = __ldg(&a.u_offset[u]);
  for (int u = threadIdx.x; u < n_u; u += kPThreads) s_slot[u] = __ldg(&a.unique_slot[u]);
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int u = 0; u < n_u; ++u) {
      s_pre[u] = acc;
      acc += (s_off[u + 1] - s_off[u] + kBM - 1) / kBM;
    }
    s_pre[n_u] = acc;
  }
  __syncthreads();
  return s_pre[n_u];
}

// The unique expert whose m-tiles contain global m-tile index mt.
__device__ __forceinline__ int tile_expert(const int* s_pre, int n_u, int mt) {
  int lo = 0, hi = n_u - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_pre[mid] <= mt) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

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
      if (idx[i] == e) {
        a.rows_by_u[p] = r0 + i;
        a.pos[r0 + i] = p;
        ++p;
      }
    carry += total;
    __syncthreads();
  }
}

// ---------------------------------------------------------------- combine
// y[t][c] = sum_{j<k} yp[pos[t*k+j]][c], four columns per thread.
__global__ void __launch_bounds__(kPThreads) combine_kernel(PrefillArgs a) {
  const int q4 = a.H / 4;
  const long long n = (long long)a.T * q4;
  for (long long i = (long long)blockIdx.x * kPThreads + threadIdx.x; i < n; i += (long long)gridDim.x * kPThreads) {
    const int t = (int)(i / q4), q = (int)(i - (long long)t * q4);
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < a.k; ++j) {
      const int p = __ldg(&a.pos[t * a.k + j]);
      const float4 v = __ldcg(reinterpret_cast<const float4*>(a.yp + (long long)p * a.H) + q);
      s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
    }
    reinterpret_cast<float4*>(a.y + (long long)t * a.H)[q] = s;
  }
}

// ---------------------------------------------------------------- gate/up
// Tile: 128 grouped rows of one expert x 64 h columns.  B holds the 64 Wg rows
// then the 64 matching Wu rows; warp (wm, wn) owns rows wm*32.. and h columns
// wn*32.. of both halves.
__global__ void __launch_bounds__(kPThreads, 2) gateup_gemm_kernel(PrefillArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  int* s_off = reinterpret_cast<int*>(smem);
  int* s_pre = s_off + (kMaxExperts + 1);
  int* s_slot = s_pre + (kMaxExperts + 1);
  __nv_bfloat16* sA = reinterpret_cast<__nv_bfloat16*>(smem + kHdrBytes);
  __nv_bfloat16* sB = sA + kStages * kTileElems;
  const int H = a.H, I = a.I, k = a.k;
  const int n_u = min(__ldg(&a.hdr[PH_UNIQUE]), kMaxExperts);
  const int mtiles = tile_table(a, n_u, s_off, s_pre, s_slot);
  const int ntiles = I / kBN1;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int wm = warp & 3, wn = warp >> 2;
  const int lrow = tid >> 2, lchunk = tid & 3;  // copy slots: rows lrow, lrow + 64; one 16-byte chunk
  const int KT = H / kBK;
  const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(a.x);
  __nv_bfloat16* h = static_cast<__nv_bfloat16*>(a.h);
  for (int tile = blockIdx.x; tile < mtiles * ntiles; tile += gridDim.x) {
    const int mt = tile / ntiles, nt = tile - mt * ntiles;
    const int u = tile_expert(s_pre, n_u, mt);
    const int p0 = s_off[u] + (mt - s_pre[u]) * kBM, pend = s_off[u + 1];
    const int n0 = nt * kBN1;
    const __nv_bfloat16* blob =
        reinterpret_cast<const __nv_bfloat16*>(a.pool + (long long)s_slot[u] * a.expert_bytes);
    const __nv_bfloat16* arow[2];
    bool aval[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {  // x rows of the tokens of grouped rows p0 + lrow + 64 i
      const int p = p0 + lrow + 64 * i;
      aval[i] = p < pend;
      const int t = aval[i] ? __ldg(&a.rows_by_u[p]) / k : 0;
      arow[i] = x + (long long)t * H + lchunk * 8;
    }
    const __nv_bfloat16* brow[2] = {blob + (long long)(n0 + lrow) * H + lchunk * 8,       // Wg
                                    blob + (long long)(I + n0 + lrow) * H + lchunk * 8};  // Wu
    auto load_stage = [&](int kt, int st) {
      __nv_bfloat16* A = sA + st * kTileElems;
      __nv_bfloat16* B = sB + st * kTileElems;
      const int k0 = kt * kBK;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        cp_async16(A + (lrow + 64 * i) * kPitch + lchunk * 8, arow[i] + k0, aval[i]);
        cp_async16(B + (lrow + 64 * i) * kPitch + lchunk * 8, brow[i] + k0, true);
      }
    };
    float accG[2][4][4], accU[2][4][4];
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
      for (int ni = 0; ni < 4; ++ni)
#pragma unroll
        for (int q = 0; q < 4; ++q) accG[mi][ni][q] = accU[mi][ni][q] = 0.0f;
#pragma unroll
    for (int st = 0; st < kStages - 1; ++st) {
      if (st < KT) load_stage(st, st);
      cp_commit();
    }
    for (int kt = 0; kt < KT; ++kt) {
      cp_wait<kStages - 2>();
      __syncthreads();  // stage kt has landed for every thread; stage kt-1 is free again
      const int nk = kt + kStages - 1;
      if (nk < KT) load_stage(nk, nk % kStages);
      cp_commit();
      const __nv_bfloat16* A = sA + (kt % kStages) * kTileElems;
      const __nv_bfloat16* B = sB + (kt % kStages) * kTileElems;
#pragma unroll
      for (int kk = 0; kk < kBK; kk += 16) {
        uint32_t af[2][4];
#pragma unroll
        for (int mi = 0; mi < 2; ++mi) ldsm_x4(af[mi], A + (wm * 32 + mi * 16 + (lane & 15)) * kPitch + kk + (lane >> 4) * 8);
#pragma unroll
        for (int nj = 0; nj < 2; ++nj) {
          const int br = wn * 32 + nj * 16 + (lane & 7) + (lane >> 4) * 8;
          const int bc = kk + ((lane >> 3) & 1) * 8;
          uint32_t bg[4], bu[4];
          ldsm_x4(bg, B + br * kPitch + bc);
          ldsm_x4(bu, B + (64 + br) * kPitch + bc);
#pragma unroll
          for (int mi = 0; mi < 2; ++mi) {
            mma_bf16(accG[mi][2 * nj], af[mi], bg[0], bg[1]);
            mma_bf16(accG[mi][2 * nj + 1], af[mi], bg[2], bg[3]);
            mma_bf16(accU[mi][2 * nj], af[mi], bu[0], bu[1]);
            mma_bf16(accU[mi][2 * nj + 1], af[mi], bu[2], bu[3]);
          }
        }
      }
    }
    cp_wait<0>();
    __syncthreads();  // every stage is free before the next tile's loads
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
      for (int ni = 0; ni < 4; ++ni)
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int p = p0 + wm * 32 + mi * 16 + (lane >> 2) + half * 8;
          if (p < pend) {
            const int c = n0 + wn * 32 + ni * 8 + (lane & 3) * 2;
            const float g0 = accG[mi][ni][2 * half], g1 = accG[mi][ni][2 * half + 1];
            const float v0 = accU[mi][ni][2 * half], v1 = accU[mi][ni][2 * half + 1];
            const __nv_bfloat162 hv =
                __floats2bfloat162_rn(g0 / (1.0f + expf(-g0)) * v0, g1 / (1.0f + expf(-g1)) * v1);
            *reinterpret_cast<__nv_bfloat162*>(h + (long long)p * I + c) = hv;
          }
        }
  }
}

// ---------------------------------------------------------------- down
// Tile: 128 grouped rows of one expert x 128 output columns; warp (wm, wn)
// owns rows wm*32.. and columns wn*64..; the gate weight of each row is
// applied in the epilogue.
__global__ void __launch_bounds__(kPThreads, 2) down_gemm_kernel(PrefillArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  int* s_off = reinterpret_cast<int*>(smem);
  int* s_pre = s_off + (kMaxExperts + 1);
  int* s_slot = s_pre + (kMaxExperts + 1);
  __nv_bfloat16* sA = reinterpret_cast<__nv_bfloat16*>(smem + kHdrBytes);
  __nv_bfloat16* sB = sA + kStages * kTileElems;
  const int H = a.H, I = a.I;
  const int n_u = min(__ldg(&a.hdr[PH_UNIQUE]), kMaxExperts);
  const int mtiles = tile_table(a, n_u, s_off, s_pre, s_slot);
  const int ntiles = H / kBN2;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int wm = warp & 3, wn = warp >> 2;
  const int lrow = tid >> 2, lchunk = tid & 3;
  const int KT = I / kBK;
  const __nv_bfloat16* h = static_cast<const __nv_bfloat16*>(a.h);
  for (int tile = blockIdx.x; tile < mtiles * ntiles; tile += gridDim.x) {
    const int mt = tile / ntiles, nt = tile - mt * ntiles;
    const int u = tile_expert(s_pre, n_u, mt);
    const int p0 = s_off[u] + (mt - s_pre[u]) * kBM, pend = s_off[u + 1];
    const int c0 = nt * kBN2;
    const __nv_bfloat16* wd =
        reinterpret_cast<const __nv_bfloat16*>(a.pool + (long long)s_slot[u] * a.expert_bytes) + 2LL * I * H;
    const __nv_bfloat16* arow[2];
    bool aval[2];
    const __nv_bfloat16* brow[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int p = p0 + lrow + 64 * i;
      aval[i] = p < pend;
      arow[i] = h + (long long)(aval[i] ? p : 0) * I + lchunk * 8;
      brow[i] = wd + (long long)(c0 + lrow + 64 * i) * I + lchunk * 8;
    }
    auto load_stage = [&](int kt, int st) {
      __nv_bfloat16* A = sA + st * kTileElems;
      __nv_bfloat16* B = sB + st * kTileElems;
      const int k0 = kt * kBK;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        cp_async16(A + (lrow + 64 * i) * kPitch + lchunk * 8, arow[i] + k0, aval[i]);
        cp_async16(B + (lrow + 64 * i) * kPitch + lchunk * 8, brow[i] + k0, true);
      }
    };
    float acc[2][8][4];
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
      for (int ni = 0; ni < 8; ++ni)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[mi][ni][q] = 0.0f;
#pragma unroll
    for (int st = 0; st < kStages - 1; ++st) {
      if (st < KT) load_stage(st, st);
      cp_commit();
    }
    for (int kt = 0; kt < KT; ++kt) {
      cp_wait<kStages - 2>();
      __syncthreads();
      const int nk = kt + kStages - 1;
      if (nk < KT) load_stage(nk, nk % kStages);
      cp_commit();
      const __nv_bfloat16* A = sA + (kt % kStages) * kTileElems;
      const __nv_bfloat16* B = sB + (kt % kStages) * kTileElems;
#pragma unroll
      for (int kk = 0; kk < kBK; kk += 16) {
        uint32_t af[2][4];
#pragma unroll
        for (int mi = 0; mi < 2; ++mi) ldsm_x4(af[mi], A + (wm * 32 + mi * 16 + (lane & 15)) * kPitch + kk + (lane >> 4) * 8);
#pragma unroll
        for (int nj = 0; nj < 4; ++nj) {
          uint32_t b[4];
          ldsm_x4(b, B + (wn * 64 + nj * 16 + (lane & 7) + (lane >> 4) * 8) * kPitch + kk + ((lane >> 3) & 1) * 8);
#pragma unroll
          for (int mi = 0; mi < 2; ++mi) {
            mma_bf16(acc[mi][2 * nj], af[mi], b[0], b[1]);
            mma_bf16(acc[mi][2 * nj + 1], af[mi], b[2], b[3]);
          }
        }
      }
    }
    cp_wait<0>();
    __syncthreads();
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int p = p0 + wm * 32 + mi * 16 + (lane >> 2) + half * 8;
        if (p < pend) {
          const float wt = __ldg(&a.topk_w[__ldg(&a.rows_by_u[p])]);
#pragma unroll
          for (int ni = 0; ni < 8; ++ni) {
            const int c = c0 + wn * 64 + ni * 8 + (lane & 3) * 2;
            *reinterpret_cast<float2*>(a.yp + (long long)p * H + c) =
                make_float2(wt * acc[mi][ni][2 * half], wt * acc[mi][ni][2 * half + 1]);
          }
        }
      }
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
  return wdtype == FT_W_BF16 && H % kBN2 == 0 && H % kBK == 0 && I % kBN1 == 0 && I % kBK == 0 &&
         E <= kMaxExperts;
}

cudaError_t launch_prefill_ffn(const PrefillArgs& a, cudaStream_t s, int* launches) {
  static std::mutex mu;
  static std::set<int> ready;  // devices whose kernel attributes are set
  int dev = 0;
  cudaError_t ge = cudaGetDevice(&dev);
  if (ge != cudaSuccess) return ge;
  std::lock_guard<std::mutex> lk(mu);
  if (!ready.count(dev)) {
    cudaError_t e = cudaFuncSetAttribute(gateup_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(down_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(gateup_gemm_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(down_gemm_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    ready.insert(dev);
  }
  const int grid = 2 * prefill_sms();
  group_rows_kernel<<<a.E, kPThreads, 0, s>>>(a);
  gateup_gemm_kernel<<<grid, kPThreads, kGemmSmem, s>>>(a);
  down_gemm_kernel<<<grid, kPThreads, kGemmSmem, s>>>(a);
  combine_kernel<<<4 * prefill_sms(), kPThreads, 0, s>>>(a);
  *launches = 4;
  return cudaGetLastError();
}

}  // namespace ft
