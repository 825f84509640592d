// Prefill-path grouped expert GEMMs on the 5th-generation tensor cores
// (tcgen05, sm_103a): the gate/up + SwiGLU GEMM and the down GEMM of the
// routed SwiGLU experts, reading the weights straight from their cache slots.
//
//   gate/up:  h[p][i]  = silu(Wg[i] . x_t) * (Wu[i] . x_t)   bf16 h, p = grouped row of (t, j)
//   down:     yp[p][c] = w_tj * (Wd[c] . h[p])               fp16 (fp32 accumulation)
//
// A tile is 128 grouped rows of one expert (M) by a block of output columns
// (N); a persistent grid walks the tiles in (m-tile, n-tile) order, m-tiles
// expert by expert.  Every CTA runs three roles:
//   warp 0      TMA producer: the A rows and the B rows of each 64-wide K
//               block into a shared-memory ring (4 stages for gate/up, 3 for
//               down, whose epilogue needs staging space), 128-byte swizzled.
//               The A rows are one 2D box of 128 grouped rows: x rows already
//               permuted into grouped order (gate/up) or h (down).  The B
//               rows come from the slot pool viewed as one 2D tensor whose
//               rows are weight rows: Wg/Wu rows for gate/up, Wd rows for down.
//   warp 1      allocates 512 TMEM columns (two 128 x 256 fp32 accumulators)
//               and one thread issues tcgen05.mma (M 128, N 256, K 16, bf16 in,
//               fp32 accumulate), four per K block; tcgen05.commit frees each
//               ring stage, and marks an accumulator full after its last block.
//   warps 2-9   epilogue: tcgen05.ld of the accumulator (warp w reads TMEM
//               lanes 32 (w % 4) .. and half of the columns; with fp8 weights
//               warps 2-5, each all the columns), SwiGLU or the gate weight;
//               gate/up writes each lane's 128-byte pieces of its h row
//               directly, down stores 32-row boxes staged in shared memory
//               with TMA; the accumulator is handed back, so the epilogue of
//               one tile overlaps the MMAs of the next.
// The gate/up B tile is 128 Wg rows followed by the same 128 Wu rows, so the
// accumulator's columns [0, 128) are gate and [128, 256) up for the same 128 h
// columns and SwiGLU needs no data exchange.
//
// fp8 weights (OCP e4m3 with one bf16 scale per 128 x 128 block): the tensor
// cores multiply 16-bit by 16-bit here, because the activations must stay
// 16-bit (e4m3 activations would put about 4% error on each dot product).
// The producer loads the fp8 B rows (64 bytes of each row per K block,
// 64-byte swizzle) into the upper half of the stage's B area, and eight
// converter warps (warps 6-13, one B row per thread) read them, multiply each
// by its block's scale (staged in shared memory once per tile; a K block of 64
// lies in one 128-wide scale block; one fp16 multiply per pair of weights
// when every scale of the tile is an fp16 value) and write fp16 into the
// 128-byte-swizzled layout the MMA reads, over the whole B area (all reads
// happen before any write: a named barrier separates them), then release the
// stage to the MMA.  fp16 rather than bf16 because an e4m3 value times a bf16
// scale has 12 significant bits: fp16 keeps 11 of them, bf16 only 8 (that
// rounding alone took the output error past the tolerance).  The activations
// of an fp8 cache are fp16 too (x is permuted into fp16 rows, h is written as
// fp16); N(0,1)-scale activations lose nothing to fp16's smaller range.
//
// Every mbarrier wait is bounded (one second of %globaltimer).  A wait that
// runs out records FT_ERR_TIMEOUT and sets a CTA-wide abort flag that ends
// every later wait at once; the producer still waits (bounded) for the copies
// it issued, the MMA thread for its MMAs, and TMEM is freed before the CTA
// exits.
//
// The grouped SwiGLU expert and its gate-weighted combine follow the routed
// experts of the MoE layers the pages serve ("FreeToken vs vLLM on one RTX
// 3090", "Why the performance differs"; the 16k-token prefill chunk of
// "FreeToken: Efficient Edge-Native MoE Serving ...", ablation paragraph).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <mutex>
#include <set>

#include "driver_api.h"
#include "ft_internal.h"

namespace ft {
namespace {

constexpr int kEpiWarps = 8;             // two per TMEM lane quarter, each taking half the columns
constexpr int kEpiWarpsFp8 = 4;          // fp8: one per TMEM lane quarter, each taking all the columns
constexpr int kCvtWarps = 8;             // fp8 weights: dequantising warps, one B row per thread
constexpr int kCvtRows = 256 / (kCvtWarps * 32);
constexpr int kTcThreads = (2 + kEpiWarps) * 32;  // producer, MMA, epilogue
constexpr int kTcThreadsFp8 = (2 + kEpiWarpsFp8 + kCvtWarps) * 32;
constexpr int kBM = 128;                 // grouped rows per tile (UMMA M)
constexpr int kBK = 64;                  // K per ring stage: one 128-byte swizzle row of bf16
constexpr int kN1 = 256;                 // gate/up UMMA N: 128 gate + 128 up columns
constexpr int kH1 = kN1 / 2;             // h columns per gate/up tile
constexpr int kAccCols = 256;            // TMEM columns per accumulator
constexpr int kTmemCols = 512;           // two accumulators
constexpr int kABytes = kBM * kBK * 2;   // 16 KB
constexpr int kBBytesMax = 256 * kBK * 2;  // 32 KB
constexpr int kStageBytes = kABytes + kBBytesMax;
constexpr int kTableInts = 3 * (kMaxExperts + 1);
constexpr unsigned long long kWaitNs = 1000000000ull;

// Dynamic shared memory: [ring (1024-aligned)][output staging][tile table][barriers][fp8 scales].
// The down GEMM's epilogue stores through staging boxes: each epilogue warp
// owns two 4 KB boxes (32 rows x 128 bytes, the layout of a 128-byte-swizzled
// TMA store box), used alternately.  The gate/up GEMM's epilogue writes its
// 128-byte pieces of h rows directly, and its ring has a stage more instead.
constexpr int kBoxBytes = 32 * 128;
constexpr int kMaxKBlocks = 128;         // fp8: K / 128 of a GEMM (hidden, inter <= 16384)
template <bool kGateUp>
struct TcLayout {
  static constexpr int kStages = kGateUp ? 4 : 3;
  static constexpr bool kStaged = !kGateUp;
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kStageOutOff = kRingBytes;
  static constexpr int kTableOff = kStageOutOff + (kStaged ? kEpiWarps * 2 * kBoxBytes : 0);
  static constexpr int kBarOff = (kTableOff + kTableInts * 4 + 15) / 16 * 16;
  static constexpr int kBarWords = 3 * kStages + 2 * 2 + 1;  // full, empty, ready, tfull, tempty, drain
  static constexpr int kScaleOff = kBarOff + kBarWords * 8 + 16;  // after the tmem holder and the abort flag
  static constexpr int kSmem = kScaleOff + 2 * kMaxKBlocks * 4 + 1024;  // + a tile's block scales, alignment slack
  static_assert(kSmem <= 227 * 1024, "shared memory of the tensor-core GEMM");
};

struct TcArgs {
  const int32_t* hdr;
  const int32_t* u_offset;     // [n_u + 1]
  const int32_t* unique_slot;  // [n_u]
  const int32_t* rows_by_u;    // [R] row ids t*k + j in grouped order
  const float* topk_w;         // [R]
  __nv_bfloat16* h;            // [R][I]
  __half* yp;                  // [R][H]
  int32_t* status;
  int H, I, k, R;
  int n_tile;                  // UMMA N of this GEMM (gate/up 256; down 256 or 128)
  long long slot_rows;         // rows of one slot in the B tensor map (3I for gate/up, 3H for down)
  const uint8_t* pool;         // fp8: the slots, for the block scales
  long long expert_bytes;
  int num_slots;
};

// ---------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t sa(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ unsigned long long now_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void bar_init(uint64_t* b, uint32_t n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(sa(b)), "r"(n) : "memory");
}
__device__ __forceinline__ bool bar_try(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(sa(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void bar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(sa(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(sa(b)) : "memory");
}
// Bounded wait; gives up at once when the CTA has aborted (unless `drain`),
// and aborts the CTA when the limit runs out.
__device__ __forceinline__ bool bwait(uint64_t* b, uint32_t parity, int32_t* status, volatile int* abort_flag,
                                      bool drain = false) {
  if (bar_try(b, parity)) return true;
  const unsigned long long t0 = now_ns();
  for (;;) {
    for (int i = 0; i < 64; ++i)
      if (bar_try(b, parity)) return true;
    if (!drain && *abort_flag) return false;
    if (now_ns() - t0 > kWaitNs) {
      if (status) atomicCAS(status, 0, (int)FT_ERR_TIMEOUT);
      *abort_flag = 1;
      return false;
    }
  }
}
__device__ __forceinline__ void tma_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
          "r"(sa(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(sa(bar))
      : "memory");
}
__device__ __forceinline__ void tma_3d(void* dst, const CUtensorMap* map, int c0, int c1, int c2, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(sa(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(sa(bar))
      : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(sa(bar))
               : "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, both K-major, described by 64-bit
// shared-memory matrix descriptors; `idesc` holds the shapes and types.
__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
      : "memory");
}
// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tc_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 2D TMA store of a shared-memory box to global coordinates (c0, c1), in the
// calling thread's bulk group.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int c0, int c1, const void* src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(sa(src))
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until at most N of the thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
// Row `row` of a 32 x 128-byte staging box in the 128-byte swizzle layout:
// 16-byte chunk i of the row sits at chunk position i ^ (row % 8).
__device__ __forceinline__ void box_put16(uint8_t* box, int row, int i, uint4 v) {
  *reinterpret_cast<uint4*>(box + row * 128 + ((i ^ (row & 7)) << 4)) = v;
}

// Shared-memory matrix descriptor of a K-major operand tile whose rows are
// 128 bytes, written by TMA with the 128-byte swizzle: 8-row groups 1024 bytes
// apart (stride byte offset), descriptor version 1, swizzle mode 128B.  The
// leading byte offset is not used by this layout.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;              // leading byte offset (16 B; unused here)
  d |= (uint64_t)(1024 >> 4) << 32;    // stride byte offset
  d |= (uint64_t)1 << 46;              // version
  d |= (uint64_t)2 << 61;              // 128-byte swizzle
  return d;
}
// Instruction descriptor, kind::f16: fp32 accumulator, A and B both bf16 (or
// both fp16), both K-major, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_16bit(int M, int N, bool bf16) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

struct Smem {
  uint8_t* ring;
  uint8_t* out;   // [kEpiWarps][2][kBoxBytes]
  int* s_off;
  int* s_pre;
  int* s_slot;
  uint64_t* full;
  uint64_t* empty;
  uint64_t* tfull;
  uint64_t* tempty;
  uint64_t* drain;
  uint64_t* ready;   // fp8: the stage's B rows are dequantised
  uint32_t* tmem_holder;
  volatile int* abort_flag;
  float* s_scale;    // fp8: the tile's block scales [2 row blocks][K / 128]
};

template <bool kGateUp>
__device__ __forceinline__ Smem carve(uint8_t* raw) {
  using L = TcLayout<kGateUp>;
  constexpr int kStages = L::kStages;
  Smem s;
  // aligned by an offset from the shared array itself (not through an integer
  // cast), so the compiler keeps every access derived from it a shared one
  uint8_t* base = raw + ((1024u - (sa(raw) & 1023u)) & 1023u);
  s.ring = base;
  s.out = base + L::kStageOutOff;
  s.s_off = reinterpret_cast<int*>(base + L::kTableOff);
  s.s_pre = s.s_off + (kMaxExperts + 1);
  s.s_slot = s.s_pre + (kMaxExperts + 1);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + L::kBarOff);
  s.full = bars;
  s.empty = bars + kStages;
  s.tfull = bars + 2 * kStages;
  s.tempty = bars + 2 * kStages + 2;
  s.drain = bars + 2 * kStages + 4;
  s.ready = bars + 2 * kStages + 5;
  s.tmem_holder = reinterpret_cast<uint32_t*>(bars + L::kBarWords);
  s.abort_flag = reinterpret_cast<volatile int*>(s.tmem_holder + 1);
  s.s_scale = reinterpret_cast<float*>(base + L::kScaleOff);
  return s;
}

// Tile table: s_off = u_offset, s_pre[u] = m-tiles of the experts before u,
// s_slot = slot of each unique expert; warp 0 scans.  Returns the m-tile total
// (0 for a plan that fails the checked builds' range checks).
__device__ int build_table(const TcArgs& a, int n_u, const Smem& s) {
  int bad = kChecked && n_u < 0;
  for (int u = threadIdx.x; u <= n_u; u += blockDim.x) {
    s.s_off[u] = __ldg(&a.u_offset[u]);
    if (kChecked) bad |= s.s_off[u] < 0 || s.s_off[u] > a.R;
  }
  for (int u = threadIdx.x; u < n_u; u += blockDim.x) {
    s.s_slot[u] = __ldg(&a.unique_slot[u]);
    if (kChecked) bad |= s.s_slot[u] < 0 || s.s_slot[u] >= a.num_slots;
  }
  if (!plan_sync(bad, a.status)) {
    __syncthreads();  // the same barrier count as the table scan below
    return 0;
  }
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int per = (n_u + 31) / 32;
    const int u0 = min(n_u, lane * per), u1 = min(n_u, u0 + per);
    int local = 0;
    for (int u = u0; u < u1; ++u) local += (s.s_off[u + 1] - s.s_off[u] + kBM - 1) / kBM;
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    int acc = incl - local;
    for (int u = u0; u < u1; ++u) {
      s.s_pre[u] = acc;
      acc += (s.s_off[u + 1] - s.s_off[u] + kBM - 1) / kBM;
    }
    if (lane == 31) s.s_pre[n_u] = incl;
  }
  __syncthreads();
  return s.s_pre[n_u];
}

__device__ __forceinline__ int tile_expert(const int* s_pre, int n_u, int mt) {
  int lo = 0, hi = n_u - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_pre[mid] <= mt) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

struct TileInfo {
  int u, p0, pend, n0, slot;
};
__device__ __forceinline__ TileInfo tile_info(const Smem& s, int n_u, int ntiles, int tile, int n_cols) {
  TileInfo t;
  const int mt = tile / ntiles, nt = tile - mt * ntiles;
  t.u = tile_expert(s.s_pre, n_u, mt);
  t.p0 = s.s_off[t.u] + (mt - s.s_pre[t.u]) * kBM;
  t.pend = s.s_off[t.u + 1];
  t.n0 = nt * n_cols;
  t.slot = s.s_slot[t.u];
  return t;
}

// One B row of a K block: 64 e4m3 weights (four 16-byte chunks of a 64-byte
// swizzled fp8 row) times their block scale, written as fp16 into row r of the
// 128-byte-swizzled 16-bit B tile.  kFast: the scale is an fp16 value, and one
// fp16 multiply per pair rounds the exact product (an e4m3 value has 4
// significant bits, the scale 8); else the product is formed in fp32 (exact)
// and rounded to fp16.  Both give the exact product rounded once to fp16.
template <bool kFast>
__device__ __forceinline__ void dequant_row(const uint4 (&raw)[4], float scl, uint8_t* B, int r) {
  const __half2 s2 = __float2half2_rn(scl);
#pragma unroll
  for (int i = 0; i < 4; ++i) {  // 16 fp8 -> 16 fp16 = two 16-byte chunks of the 16-bit row
    const uint32_t w4[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
    uint32_t o[8];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w4[q] & 0xffffu), __NV_E4M3);
      const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w4[q] >> 16), __NV_E4M3);
      __half2 ha, hb;
      if (kFast) {
        ha = __hmul2(__half2(lo), s2);
        hb = __hmul2(__half2(hi), s2);
      } else {
        const float2 fa = __half22float2(__half2(lo)), fb = __half22float2(__half2(hi));
        ha = __floats2half2_rn(fa.x * scl, fa.y * scl);
        hb = __floats2half2_rn(fb.x * scl, fb.y * scl);
      }
      o[2 * q] = *reinterpret_cast<const uint32_t*>(&ha);
      o[2 * q + 1] = *reinterpret_cast<const uint32_t*>(&hb);
    }
    const int j0 = 2 * i, j1 = 2 * i + 1;
    *reinterpret_cast<uint4*>(B + r * 128 + ((j0 ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
    *reinterpret_cast<uint4*>(B + r * 128 + ((j1 ^ (r & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

// kGateUp: the gate/up + SwiGLU GEMM (A = grouped x rows, B = Wg/Wu rows);
// else the down GEMM (A = h rows, B = Wd rows).  map_a and map_b load boxes of
// 64 columns x 128 rows (x, h, Wg/Wu) or N rows (Wd); map_out stores 32-row
// output boxes.
template <bool kGateUp, bool kFp8>
__global__ void __launch_bounds__(kFp8 ? kTcThreadsFp8 : kTcThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                   const __grid_constant__ CUtensorMap map_out, TcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  constexpr int kStages = TcLayout<kGateUp>::kStages;
  const Smem s = carve<kGateUp>(smem_raw);
  constexpr int kEpi = kFp8 ? kEpiWarpsFp8 : kEpiWarps;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_u = min(__ldg(&a.hdr[PH_UNIQUE]), kMaxExperts);
  const int N = kGateUp ? kN1 : a.n_tile;           // UMMA N
  const int n_cols = kGateUp ? kH1 : a.n_tile;      // output columns per tile
  const int ntiles = (kGateUp ? a.I : a.H) / n_cols;
  const int KT = (kGateUp ? a.H : a.I) / kBK;
  const uint32_t b_bytes = (uint32_t)N * kBK * (kFp8 ? 1 : 2);  // bytes the producer loads into the B area

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      bar_init(&s.full[i], 1);
      bar_init(&s.empty[i], 1);
      bar_init(&s.ready[i], kCvtWarps);
    }
    for (int i = 0; i < 2; ++i) {
      bar_init(&s.tfull[i], 1);
      bar_init(&s.tempty[i], kEpi);
    }
    bar_init(s.drain, 1);
    *s.abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {  // the whole warp allocates the two accumulators
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(sa(s.tmem_holder)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    tc_fence_before();
  }
  const int mtiles = build_table(a, n_u, s);  // contains __syncthreads: barriers and TMEM base are visible after it
  tc_fence_after();
  const uint32_t tmem = *s.tmem_holder;
  const int total = mtiles * ntiles;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_a)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_b)) : "memory");
    }
    int it = 0;
    bool go = true;
    for (int tile = blockIdx.x; tile < total && go; tile += gridDim.x) {
      const TileInfo t = tile_info(s, n_u, ntiles, tile, n_cols);
      const long long brow = (long long)t.slot * a.slot_rows + (kGateUp ? t.n0 : 2LL * a.H + t.n0);
      for (int kt = 0; kt < KT; ++kt, ++it) {
        const int st = it % kStages;
        bool ok = true;
        if (lane == 0) ok = bwait(&s.empty[st], ((it / kStages) & 1) ^ 1, a.status, s.abort_flag);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
          go = false;
          break;
        }
        bar_try(&s.empty[st], ((it / kStages) & 1) ^ 1);  // every lane observes the freed stage itself
        uint8_t* A = s.ring + st * kStageBytes;
        uint8_t* B = A + kABytes;
        if (lane == 0) bar_expect_tx(&s.full[st], kABytes + b_bytes);
        __syncwarp();
        const int c0 = kt * kBK;
        if (lane == 0) {
          tma_2d(A, &map_a, c0, t.p0, &s.full[st]);                              // 128 grouped x or h rows
          if (kFp8) {  // fp8 rows (64 bytes of each per K block) into the upper half of the B area
            uint8_t* B8 = B + kBBytesMax / 2;
            if (kGateUp) {
              tma_3d(B8, &map_b, c0, t.n0, t.slot, &s.full[st]);                 // 128 Wg rows
              tma_3d(B8 + kBM * 64, &map_b, c0, a.I + t.n0, t.slot, &s.full[st]);  // the same Wu rows
            } else {
              tma_3d(B8, &map_b, c0, t.n0, t.slot, &s.full[st]);                 // N Wd rows
            }
          } else {
            tma_2d(B, &map_b, c0, (int)brow, &s.full[st]);                       // 128 Wg rows / N Wd rows
            if (kGateUp) tma_2d(B + kBM * 128, &map_b, c0, (int)(brow + a.I), &s.full[st]);  // the same Wu rows
          }
        }
      }
    }
    // no copy may still be writing this CTA's shared memory when it exits
    if (lane == 0)
      for (int j = it - kStages < 0 ? 0 : it - kStages; j < it; ++j)
        bwait(&s.full[j % kStages], (j / kStages) & 1, a.status, s.abort_flag, true);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_16bit(kBM, N, !kFp8);
      int it = 0, j = 0;
      bool go = true;
      for (int tile = blockIdx.x; tile < total && go; tile += gridDim.x, ++j) {
        const int acc = j & 1;
        if (!bwait(&s.tempty[acc], ((j >> 1) & 1) ^ 1, a.status, s.abort_flag)) break;
        tc_fence_after();
        const uint32_t d = tmem + acc * kAccCols;
        for (int kt = 0; kt < KT; ++kt, ++it) {
          const int st = it % kStages;
          if (!bwait(kFp8 ? &s.ready[st] : &s.full[st], (it / kStages) & 1, a.status, s.abort_flag)) {
            go = false;
            break;
          }
          if (kFp8) bar_try(&s.full[st], (it / kStages) & 1);  // the A box landed too
          tc_fence_after();
          const uint32_t A = sa(s.ring + st * kStageBytes), B = A + kABytes;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)  // K 16 per MMA: 32 bytes along the swizzled row
            tc_mma(d, sw128_desc(A + kk * 32), sw128_desc(B + kk * 32), idesc, (kt | kk) != 0);
          tc_commit(&s.empty[st]);  // the stage is free once these MMAs have read it
        }
        if (go) tc_commit(&s.tfull[acc]);
      }
      // every MMA this thread issued has completed before TMEM is freed
      tc_commit(s.drain);
      bwait(s.drain, 0, a.status, s.abort_flag, true);
    }
    __syncwarp();
  } else if (kFp8 && warp >= 2 + kEpi) {
    // ------------------------------------------------------------ fp8 dequantising warps
    if (kFp8) {
      const int ctid = threadIdx.x - (2 + kEpi) * 32;  // B rows ctid + h * (kCvtWarps * 32)
      const long long scale_off = 3LL * a.H * a.I;
      const int hb = a.H / 128, ib = a.I / 128;
      int it = 0;
      bool go = true;
      for (int tile = blockIdx.x; tile < total && go; tile += gridDim.x) {
        const TileInfo t = tile_info(s, n_u, ntiles, tile, n_cols);
        const uint16_t* sc = reinterpret_cast<const uint16_t*>(a.pool + (long long)t.slot * a.expert_bytes + scale_off);
        // the tile's block scales, one per (128-row block, 128-wide K block), read
        // from the slot once per tile instead of once per stage and row
        const int KB = KT / 2;
        asm volatile("bar.sync 5, %0;" ::"n"(kCvtWarps * 32) : "memory");  // the previous tile's are read
        uint32_t inexact = 0;
        for (int i = ctid; i < 2 * KB; i += kCvtWarps * 32) {
          const int rb = i / KB, kb = i - rb * KB;
          float v = 0.0f;
          if (rb * kBM < N) {
            const int idx = kGateUp ? (rb ? ib * hb : 0) + (t.n0 >> 7) * hb + kb  // Wg, then Wu row blocks
                                    : 2 * ib * hb + ((t.n0 >> 7) + rb) * ib + kb;  // Wd row blocks
            v = __uint_as_float((uint32_t)__ldg(sc + idx) << 16);
          }
          s.s_scale[i] = v;
          inexact |= __half2float(__float2half_rn(v)) != v;
        }
        // fast: every block scale of the tile is an fp16 value (a bf16 scale
        // below 2^-14 or beyond fp16's range is not, and takes the fp32 route)
        uint32_t fast;
        asm volatile(
            "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\tbar.red.or.pred p, 5, %2, q;\n\t"
            "selp.u32 %0, 0, 1, p;\n\t}"
            : "=r"(fast)
            : "r"(inexact), "n"(kCvtWarps * 32)
            : "memory");
        for (int kt = 0; kt < KT; ++kt, ++it) {
          const int st = it % kStages;
          bool ok = true;
          if (lane == 0) ok = bwait(&s.full[st], (it / kStages) & 1, a.status, s.abort_flag);
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (ok) bar_try(&s.full[st], (it / kStages) & 1);
          uint8_t* B = s.ring + st * kStageBytes + kABytes;
          const uint8_t* B8 = B + kBBytesMax / 2;
          const int kb = (kt * kBK) >> 7;  // the 128-wide K block of this stage
          uint4 raw[kCvtRows][4];
          float scl[kCvtRows];
#pragma unroll
          for (int h = 0; h < kCvtRows; ++h) {
            const int r = ctid + h * (kCvtWarps * 32);
            scl[h] = 0.0f;
            if (ok && r < N) {
#pragma unroll
              for (int i = 0; i < 4; ++i)  // 64-byte-swizzled fp8 row r
                raw[h][i] = *reinterpret_cast<const uint4*>(B8 + r * 64 + ((i ^ ((r >> 1) & 3)) << 4));
              scl[h] = s.s_scale[(r >> 7) * KB + kb];  // gate/up: rows < 128 are Wg rows; down: rows n0 + r
            }
          }
          // every fp8 row is read before any 16-bit row is written; the four warps
          // agree on stopping (a wait that ran out anywhere) at the same barrier
          uint32_t stop;
          asm volatile(
              "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\tbar.red.or.pred p, 4, %2, q;\n\t"
              "selp.u32 %0, 1, 0, p;\n\t}"
              : "=r"(stop)
              : "r"((uint32_t)(!ok || *s.abort_flag)), "n"(kCvtWarps * 32)
              : "memory");
          if (stop) {
            go = false;
            break;
          }
#pragma unroll
          for (int h = 0; h < kCvtRows; ++h) {
            const int r = ctid + h * (kCvtWarps * 32);
            if (r < N) {
              if (fast) dequant_row<true>(raw[h], scl[h], B, r);
              else dequant_row<false>(raw[h], scl[h], B, r);
            }
          }
          fence_async_smem();  // the tensor core reads these rows through the async proxy
          __syncwarp();
          if (lane == 0) bar_arrive(&s.ready[st]);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Warp w reads TMEM lanes 32 (w % 4) .. (the tile's rows 32 q ..) and half
    // of the tile's columns.  A 32-row group that lies wholly before the
    // expert's last row goes out through a swizzled staging box and one TMA
    // store (full 128-byte lines); a group cut by the expert's end is stored
    // row by row by its live lanes, so no store touches the next expert's rows.
    const int q = warp & 3;                     // TMEM lanes 32q .. 32q + 31
    uint8_t* boxes = s.out + (warp - 2) * 2 * kBoxBytes;
    int nbox = 0;
    int j = 0;
    auto next_box = [&]() -> uint8_t* {          // a staging box no earlier store still reads
      uint8_t* b = boxes + (nbox & 1) * kBoxBytes;
      ++nbox;
      if (lane == 0) bulk_wait_read<1>();
      __syncwarp();
      return b;
    };
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++j) {
      const int acc = j & 1;
      bool ok = true;
      if (lane == 0) ok = bwait(&s.tfull[acc], (j >> 1) & 1, a.status, s.abort_flag);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      bar_try(&s.tfull[acc], (j >> 1) & 1);  // every lane observes the completed phase itself
      tc_fence_after();
      const TileInfo t = tile_info(s, n_u, ntiles, tile, n_cols);
      const int r0 = t.p0 + q * 32;              // first grouped row of this warp's group
      const int live_rows = min(32, max(0, t.pend - r0));
      const bool live = lane < live_rows;
      const bool boxed = TcLayout<kGateUp>::kStaged && live_rows == 32;
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + acc * kAccCols;
      for (int hh = 0; hh < (kEpi == 8 ? 1 : 2) && live_rows > 0; ++hh) {
        const int half = kEpi == 8 ? (warp - 2) >> 2 : hh;  // which half of the columns
        if (kGateUp) {
          // h columns [hc, hc + 64): gate at TMEM columns hc.., up at kH1 + hc..
          const int hc = half * 64;
          uint8_t* box = boxed ? next_box() : nullptr;
          __nv_bfloat16* hrow = a.h + (long long)(r0 + lane) * a.I + t.n0 + hc;
          for (int c = 0; c < 64; c += 32) {
            float g[32], u[32];
            tc_ld32(tbase + hc + c, g);
            tc_ld32(tbase + kH1 + hc + c, u);
            uint32_t packed[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {  // silu(g) * u = g u / (1 + e^-g); h is rounded to bf16 (fp16)
              const float h0 = __fdividef(g[2 * i] * u[2 * i], 1.0f + __expf(-g[2 * i]));
              const float h1 = __fdividef(g[2 * i + 1] * u[2 * i + 1], 1.0f + __expf(-g[2 * i + 1]));
              if (kFp8) {
                const __half2 hv = __floats2half2_rn(h0, h1);
                packed[i] = *reinterpret_cast<const uint32_t*>(&hv);
              } else {
                const __nv_bfloat162 hv = __floats2bfloat162_rn(h0, h1);
                packed[i] = *reinterpret_cast<const uint32_t*>(&hv);
              }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint4 v = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
              if (boxed) box_put16(box, lane, (c >> 3) + i, v);
              else if (live) reinterpret_cast<uint4*>(hrow + c)[i] = v;
            }
          }
          if (boxed) {
            fence_async_smem();
            __syncwarp();
            if (lane == 0) tma_store_2d(&map_out, t.n0 + hc, r0, box);
          }
        } else {
          // output columns [t.n0 + half * n_cols / 2, ...) in chunks of 64, rounded to fp16
          const float wt = live ? __ldg(&a.topk_w[__ldg(&a.rows_by_u[r0 + lane])]) : 0.0f;
          const int cw = n_cols / 2;
          __half* yrow = a.yp + (long long)(r0 + lane) * a.H + t.n0 + half * cw;
          for (int c = 0; c < cw; c += 64) {
            float v[64];
            tc_ld32(tbase + half * cw + c, v);
            tc_ld32(tbase + half * cw + c + 32, v + 32);
            uint8_t* box = boxed ? next_box() : nullptr;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              uint32_t w4[4];
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const __half2 hv = __floats2half2_rn(wt * v[8 * i + 2 * q], wt * v[8 * i + 2 * q + 1]);
                w4[q] = *reinterpret_cast<const uint32_t*>(&hv);
              }
              const uint4 u = make_uint4(w4[0], w4[1], w4[2], w4[3]);
              if (boxed) box_put16(box, lane, i, u);
              else if (live) reinterpret_cast<uint4*>(yrow + c)[i] = u;
            }
            if (boxed) {
              fence_async_smem();
              __syncwarp();
              if (lane == 0) tma_store_2d(&map_out, t.n0 + half * cw + c, r0, box);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) bar_arrive(&s.tempty[acc]);  // this warp's part of the accumulator is read
    }
    if (lane == 0) bulk_wait_all();  // every TMA store of this warp has completed
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// A 2D tensor map, `cols` x `rows` (cols innermost, row pitch `pitch`
// bytes), box `box_cols` x `box_rows`, 128-byte swizzle, zero fill outside.
cudaError_t tmap_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, unsigned long long cols,
                    unsigned long long rows, unsigned long long pitch, uint32_t box_cols, uint32_t box_rows) {
  static EncodeTiled enc = nullptr;
  if (!enc) enc = reinterpret_cast<EncodeTiled>(driver_fn("cuTensorMapEncodeTiled"));
  if (!enc) return cudaErrorNotSupported;
  if ((reinterpret_cast<uintptr_t>(base) & 15) || (pitch & 15)) return cudaErrorInvalidValue;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {pitch};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}
cudaError_t bf16_map(CUtensorMap* m, const void* base, unsigned long long cols, unsigned long long rows,
                     unsigned long long pitch, uint32_t box_cols, uint32_t box_rows) {
  return tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, cols, rows, pitch, box_cols, box_rows);
}

int tc_sms() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
  }
  return n;
}

}  // namespace

bool prefill_tc_supported(int H, int I) {
  return H % 128 == 0 && I % kH1 == 0 && H % kBK == 0 && I % kBK == 0 && H <= 128 * kMaxKBlocks &&
         I <= 128 * kMaxKBlocks;
}

// A 3D byte tensor map over rows of the slot pool: [slot][row < rows][cols
// bytes] starting `offset` bytes into each slot, boxes of 64 bytes x box_rows
// rows x 1 slot, 64-byte swizzle (the fp8 weight rows of a K block).
cudaError_t fp8_rows_map(CUtensorMap* m, const uint8_t* pool, long long offset, unsigned long long cols,
                         unsigned long long rows, int num_slots, long long expert_bytes, uint32_t box_rows) {
  static EncodeTiled enc = nullptr;
  if (!enc) enc = reinterpret_cast<EncodeTiled>(driver_fn("cuTensorMapEncodeTiled"));
  if (!enc) return cudaErrorNotSupported;
  const uint8_t* base = pool + offset;
  if ((reinterpret_cast<uintptr_t>(base) & 15) || (expert_bytes & 15) || (cols & 15)) return cudaErrorInvalidValue;
  const cuuint64_t dims[3] = {cols, rows, (cuuint64_t)num_slots};
  const cuuint64_t strides[2] = {cols, (cuuint64_t)expert_bytes};
  const cuuint32_t box[3] = {64, box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <bool kGateUp, bool kFp8>
cudaError_t set_smem_attr() {
  return cudaFuncSetAttribute(tc_gemm_kernel<kGateUp, kFp8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              TcLayout<kGateUp>::kSmem);
}

cudaError_t launch_prefill_gemms(const PrefillArgs& p, int num_slots, cudaStream_t st, const cudaEvent_t* marks) {
  static std::mutex mu;
  static std::set<int> ready;  // devices whose kernel attributes are set
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (!ready.count(dev)) {
      e = set_smem_attr<true, false>();
      if (e == cudaSuccess) e = set_smem_attr<false, false>();
      if (e == cudaSuccess) e = set_smem_attr<true, true>();
      if (e == cudaSuccess) e = set_smem_attr<false, true>();
      if (e != cudaSuccess) return e;
      ready.insert(dev);
    }
  }
  const bool fp8 = p.wdtype == FT_W_FP8E4M3_B128;
  if (!fp8 && p.wdtype != FT_W_BF16) return cudaErrorNotSupported;
  const int H = p.H, I = p.I, R = p.T * p.k;
  TcArgs a{};
  a.hdr = p.hdr; a.u_offset = p.u_offset; a.unique_slot = p.unique_slot; a.rows_by_u = p.rows_by_u;
  a.topk_w = p.topk_w; a.h = static_cast<__nv_bfloat16*>(p.h); a.yp = static_cast<__half*>(p.yp); a.status = p.status;
  a.H = H; a.I = I; a.k = p.k; a.R = R;
  a.pool = p.pool; a.expert_bytes = p.expert_bytes; a.num_slots = num_slots;
  CUtensorMap mx, mw1, mh, mwd, mh_out, myp_out;
  // xp [R][H]: the x rows in grouped order
  if ((e = bf16_map(&mx, p.xp, H, R, 2ull * H, kBK, kBM)) != cudaSuccess) return e;
  // h [R][I]
  if ((e = bf16_map(&mh, p.h, I, R, 2ull * I, kBK, kBM)) != cudaSuccess) return e;
  const int n2 = H % 256 == 0 ? 256 : 128;
  if (fp8) {
    // Wg, Wu rows of every slot: [slot][2I rows][H bytes]; Wd rows: [slot][H rows][I bytes]
    if ((e = fp8_rows_map(&mw1, p.pool, 0, H, 2ull * I, num_slots, p.expert_bytes, kBM)) != cudaSuccess) return e;
    if ((e = fp8_rows_map(&mwd, p.pool, 2LL * H * I, I, H, num_slots, p.expert_bytes, n2)) != cudaSuccess) return e;
  } else {
    // the pool as rows of H: Wg rows [s*3I, s*3I + I), Wu rows [s*3I + I, s*3I + 2I)
    if ((e = bf16_map(&mw1, p.pool, H, 3ull * I * num_slots, 2ull * H, kBK, kBM)) != cudaSuccess) return e;
    // the pool as rows of I: Wd rows [s*3H + 2H, s*3H + 3H)
    if ((e = bf16_map(&mwd, p.pool, I, 3ull * H * num_slots, 2ull * I, kBK, n2)) != cudaSuccess) return e;
  }
  // output boxes of 32 rows x 128 bytes: h (64 bf16 columns) and yp (64 fp16 columns)
  if ((e = bf16_map(&mh_out, p.h, I, R, 2ull * I, 64, 32)) != cudaSuccess) return e;
  if ((e = tmap_2d(&myp_out, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, p.yp, H, R, 2ull * H, 64, 32)) != cudaSuccess) return e;
  const int grid = tc_sms();
  const int threads = fp8 ? kTcThreadsFp8 : kTcThreads;
  a.n_tile = kN1;
  a.slot_rows = 3LL * I;
  if (marks && (e = cudaEventRecord(marks[0], st)) != cudaSuccess) return e;
  constexpr int kSmem1 = TcLayout<true>::kSmem, kSmem2 = TcLayout<false>::kSmem;
  if (fp8) tc_gemm_kernel<true, true><<<grid, threads, kSmem1, st>>>(mx, mw1, mh_out, a);
  else tc_gemm_kernel<true, false><<<grid, threads, kSmem1, st>>>(mx, mw1, mh_out, a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (marks && (e = cudaEventRecord(marks[1], st)) != cudaSuccess) return e;
  a.n_tile = n2;
  a.slot_rows = 3LL * H;
  if (marks && (e = cudaEventRecord(marks[2], st)) != cudaSuccess) return e;
  if (fp8) tc_gemm_kernel<false, true><<<grid, threads, kSmem2, st>>>(mh, mwd, myp_out, a);
  else tc_gemm_kernel<false, false><<<grid, threads, kSmem2, st>>>(mh, mwd, myp_out, a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (marks && (e = cudaEventRecord(marks[3], st)) != cudaSuccess) return e;
  return cudaSuccess;
}

}  // namespace ft
