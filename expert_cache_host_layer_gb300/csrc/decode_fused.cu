// Decode-path expert FFN (T <= 8 tokens) as one kernel per layer that streams
// every weight byte once and needs no grid-wide barrier:
//
//   y[t] = sum over the picks (t, j) of w_tj * Wd_e h,   h = silu(Wg_e x_t) * (Wu_e x_t)
//
// The work is cut into units of R consecutive intermediate rows of one unique
// expert, R chosen so that one Wd row's slice of the unit is 64 bytes (32
// bf16, 64 fp8, 16 fp32).  A CTA (one per SM) takes units round-robin; for a
// unit it
//   phase A   streams the unit's R Wg rows and R Wu rows (contiguous in the
//             slot) through a 4-stage shared-memory ring with bulk copies and
//             computes h' = w_tj * silu(g) * u for the expert's tokens into
//             shared memory (consumer warps take row pairs round-robin);
//   phase B   streams the unit's columns of Wd - the 64-byte slice of every
//             one of the H rows - as 3D TMA boxes of 256 rows (64-byte
//             swizzle), and each consumer thread owns one output row c of a
//             box: it dots the slice with h' of each token and adds the result
//             into y[t][c] with a fp32 reduction in global memory.
// So the down projection of a unit needs only that unit's h: there is no
// exchange of h between CTAs and no grid barrier.  y is zeroed once per
// launch by CTA 0, which then sets a flag to the launch's event number; the
// other CTAs wait (bounded) for that value before their first addition, long
// after it is set.
// The additions into y from different units arrive in no fixed order, so y
// is reproducible only to fp32 rounding.
//
// The kernel is launched as a programmatic dependent of the kernel before it
// on the stream: its barrier set-up, plan staging and the first bulk copies
// of a hit expert's rows overlap the end of the previous layer's FFN;
// griddepcontrol.wait precedes every read of a missed expert's slot, x and y.
//
// Up to four more warps per CTA copy the NEXT layer's missed blobs from the
// host bank (mapped pinned memory, read over the host link) into their victim
// slots while this layer's experts stream from HBM (SM-pull mode).  The
// victims exclude this layer's slots (pin rule) and the previous layer's FFN
// has finished (griddepcontrol.wait), so nothing still reads them.
//
// Every wait is bounded (about one second of %globaltimer); a wait that runs
// out records FT_ERR_TIMEOUT in the status word and sets a CTA-wide abort
// flag that ends later waits at once; the producer still waits (bounded) for
// the copies it issued before the CTA exits.
//
// The SwiGLU expert and its gate-weighted combine follow the routed experts
// of the Qwen3-MoE / DeepSeek MoE layers the pages serve ("FreeToken vs vLLM
// on one RTX 3090", "Why the performance differs"; "FreeToken: Efficient
// Edge-Native MoE Serving ...", design paragraph: the FFN reads experts from
// the GPU expert cache; ablation paragraph: the next layer's experts are
// transferred while this layer computes).
#include <cuda.h>

#include <map>
#include <mutex>

#include "decode_common.h"
#include "driver_api.h"
#include "ft_internal.h"

namespace ft {
namespace {
using namespace dec;

constexpr int kCons = 8;                                   // consumer warps
constexpr int kCopyWarps = kMaxFetchWarps;                 // next-layer copy warps
constexpr int kThreadsF = (kCons + 1 + kCopyWarps) * 32;   // + one producer warp
constexpr int kStagesF = 4;
constexpr int kStageF = 32 * 1024;
constexpr int kBoxRows = kCons * 32;                       // Wd rows per TMA box: one per consumer thread
constexpr int kSlice = 64;                                 // bytes of one Wd row in a unit
constexpr int kBoxBytes = kBoxRows * kSlice;               // 16 KB
constexpr int kCopyUnroll = 8;                             // 16-byte loads in flight per copy thread
constexpr int kMaxT = kDecodeMaxTokens;

__host__ __device__ __forceinline__ int up(int v, int a) { return (v + a - 1) / a * a; }

struct Lay {
  int R, P, x_off, plan_off, w_off, hs_off, sc_off, bar_off, ring_off, total;
  __host__ __device__ Lay(int H, int I, int T, int wsize, int act_bytes, int max_unique, int rows) {
    R = kSlice / wsize;
    P = kStageF / (2 * H * wsize);  // row pairs (a Wg row and its Wu row) per phase-A stage
    if (P > R) P = R;
    x_off = 0;
    plan_off = up(T * H * act_bytes, 16);
    w_off = plan_off + up((2 * max_unique + 1 + rows) * 4, 16);  // unique_slot, u_offset, rows_by_u
    hs_off = w_off + up(rows * 4, 16);
    sc_off = hs_off + up(kMaxT * R * 4, 16);
    bar_off = sc_off + (wsize == 1 ? up(3 * (H / 128) * 4, 16) : 0);  // fp8: the unit's block scales
    ring_off = up(bar_off + (2 * kStagesF + 2) * 8, 1024);
    total = ring_off + kStagesF * kStageF + 1024;  // + slack to align the ring to 1024 bytes
  }
  __host__ __device__ bool ok(int H, int I, int wsize) const {
    return P >= 1 && R % P == 0 && I % R == 0 && H % kBoxRows == 0;
  }
};

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
// Lane 0 waits, then every lane observes the completed phase itself (so the
// async-proxy writes are visible to it).
__device__ __forceinline__ bool acquire(uint64_t* full, uint32_t parity, int32_t* status, volatile int* abort_flag) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = fwait(full, parity, status, abort_flag);
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok) mbar_try_wait(full, parity);
  return ok;
}
__device__ __forceinline__ void release(uint64_t* empty) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(empty);
}
__device__ __forceinline__ void cons_sync() { asm volatile("bar.sync 3, %0;" ::"n"(kCons * 32) : "memory"); }

__device__ __forceinline__ void tma_3d(void* dst, const CUtensorMap* map, int c0, int c1, int c2, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ uint4 ld_host16(const uint4* p) {  // streamed once: evict first
  uint4 v;
  asm volatile("ld.global.cs.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// The copy warps' work: 16-byte words of the next event's missed blobs, in
// items of nw * 32 * kCopyUnroll words (nw copy warps take part), item i on
// CTA i % grid.
__device__ __forceinline__ void copy_next_misses(const PullArgs& p, int ct, int nw) {
  const long long kItem16 = (long long)nw * 32 * kCopyUnroll;
  int n_miss = __ldcg(&p.hdr[PH_MISS]);
  if (!checked_ok(n_miss >= 0 && n_miss <= p.E, p.status)) n_miss = 0;
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
    if (!checked_ok(slot >= 0 && slot < p.num_slots && e >= 0 && e < p.E, p.status)) continue;
    const long long blob = ((long long)p.layer * p.E + e) % p.bank_blobs;
    const uint4* src = bank + blob * eb16 + c * kItem16;
    uint4* dst = pool + (long long)slot * eb16 + c * kItem16;
    const long long n = min(kItem16, eb16 - c * kItem16);
    uint4 v[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const long long i = (long long)u * (nw * 32) + ct;
      if (i < n) v[u] = ld_host16(src + i);
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const long long i = (long long)u * (nw * 32) + ct;
      if (i < n) dst[i] = v[u];
    }
  }
}

// 16-byte chunk i (0..3) of row r of a 64-byte-swizzled box of 64-byte rows.
__device__ __forceinline__ uint4 box_get16(const uint8_t* box, int r, int i) {
  return *reinterpret_cast<const uint4*>(box + r * kSlice + ((i ^ ((r >> 1) & 3)) << 4));
}

// MR: rows (tokens) of one expert handled together: 1 for single-token
// decode, else 4; an expert with more rows (T up to 8) takes a second pass
// over the staged weights, so a batch of a few tokens does not carry eight
// rows' registers and predicates.
// NCL: 16-byte chunks per lane of one Wg/Wu row (the row's chunks <= 32 NCL),
// so the phase-A dot products unroll fully and every lane has NCL chunks of
// loads in flight.
template <int WT, int MR, int NCL>
__global__ void __maxnreg__(96) ffn_fused_kernel(const __grid_constant__ CUtensorMap wd_map, FfnArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  constexpr bool kF32 = WT == FT_W_F32;
  constexpr int EPC = W<WT>::kEPC, WSZ = W<WT>::kBytes;
  constexpr int R = kSlice / WSZ;
  const int H = a.H, I = a.I, k = a.k, T = a.T;
  const int act_bytes = kF32 ? 4 : 2;
  const int rows_total = T * k;
  const Lay lay(H, I, T, WSZ, act_bytes, a.max_unique, rows_total);
  const int P = lay.P;
  uint8_t* xs = smem + lay.x_off;
  int32_t* p_slot = reinterpret_cast<int32_t*>(smem + lay.plan_off);
  int32_t* p_off = p_slot + a.max_unique;
  int32_t* p_rows = p_off + a.max_unique + 1;
  float* p_w = reinterpret_cast<float*>(smem + lay.w_off);
  float* hs = reinterpret_cast<float*>(smem + lay.hs_off);  // [MR][R] h' of the current unit
  float* s_sc = reinterpret_cast<float*>(smem + lay.sc_off);  // fp8: [Wg | Wu | Wd] block scales of the unit
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + lay.bar_off);
  uint64_t* empty = full + kStagesF;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kStagesF);
  // 1024-aligned by an offset from the shared array (not through an integer
  // cast), so the compiler keeps the ring's loads shared-memory loads
  uint8_t* ring = smem + lay.ring_off + ((1024u - (smem_addr(smem + lay.ring_off) & 1023u)) & 1023u);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_u = min(__ldg(&a.hdr[PH_UNIQUE]), a.max_unique);
  const long long row_g = (long long)H * WSZ;
  const long long scale_off = 3LL * H * I * WSZ;
  const int upe = I / R;  // units per expert
  const int n_boxes = H / kBoxRows;
  const int event = __ldg(&a.hdr[PH_EVENT]);
  unsigned* done_ctr = a.gbar + 2;
  unsigned* y_flag = a.gbar + 3;

  // ---- prologue: may overlap the end of the previous kernel on the stream
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesF; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kCons);
    }
    *abort_flag = 0;
    mbar_init_fence();
  }
  int bad = 0;  // checked builds: a plan index out of range
  for (int i = threadIdx.x; i < n_u; i += kThreadsF) {
    p_slot[i] = __ldg(&a.unique_slot[i]);
    if (kChecked) bad |= p_slot[i] < 0 || p_slot[i] >= a.num_slots;
  }
  for (int i = threadIdx.x; i <= n_u; i += kThreadsF) {
    p_off[i] = __ldg(&a.u_offset[i]);
    if (kChecked) bad |= p_off[i] < 0 || p_off[i] > rows_total;
  }
  for (int i = threadIdx.x; i < rows_total; i += kThreadsF) {
    p_rows[i] = __ldg(&a.rows_by_u[i]);
    p_w[i] = __ldg(&a.topk_w[i]);
    if (kChecked) bad |= p_rows[i] < 0 || p_rows[i] >= rows_total;
  }
  // a bad plan is reported and computes nothing (the copy warps check their own indices)
  const int n_units = plan_sync(bad, a.status) ? n_u * upe : 0;
  // The first unit's Wg/Wu rows start streaming before the previous kernel is
  // known to be complete when its expert was a hit: nothing writes a hit's
  // slot now (the copies of this event go to its misses' victims; those of
  // earlier events finished before the kernel before this one passed its own
  // griddepcontrol.wait, which precedes its launch_dependents).
  int i_pre = 0;
  if (threadIdx.x == kCons * 32 && a.hit && (int)blockIdx.x < n_units) {
    const int u = blockIdx.x / upe;
    if (__ldg(&a.hit[u])) {
      const int r0 = (blockIdx.x - u * upe) * R;
      const uint8_t* blob = a.pool + (long long)p_slot[u] * a.expert_bytes;
      const uint32_t b = (uint32_t)(P * row_g);
      for (int r = r0; r < r0 + R && i_pre < kStagesF; r += P, ++i_pre) {
        mbar_expect_tx(&full[i_pre], 2 * b);
        bulk_g2s(ring + (size_t)i_pre * kStageF, blob + r * row_g, b, &full[i_pre]);
        bulk_g2s(ring + (size_t)i_pre * kStageF + b, blob + ((long long)I + r) * row_g, b, &full[i_pre]);
      }
    }
  }
  pdl_wait_primary();       // the previous kernel (and every slot write it made) is complete
  pdl_launch_dependents();  // the next layer's FFN may queue up behind this one
  {
    const int n16 = T * H * act_bytes / 16;
    const uint4* src = static_cast<const uint4*>(a.x);
    for (int i = threadIdx.x; i < n16; i += kThreadsF) reinterpret_cast<uint4*>(xs)[i] = src[i];
  }
  __syncthreads();

  // ---- copy warps: the next layer's misses
  if (warp > kCons) {
    const int nw = min(max(a.fetch_warps, 1), kCopyWarps);
    if (a.nx.hdr && warp - (kCons + 1) < nw) copy_next_misses(a.nx, threadIdx.x - (kCons + 1) * 32, nw);
    return;
  }

  // ---- producer
  if (warp == kCons) {
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&wd_map)) : "memory");
      wait_ready_flag(a);  // copy-engine mode: the slots' bytes are in place
      int i = 0;
      bool go = true;
      auto stage_free = [&](int s) -> bool {
        return i < kStagesF || fwait(&empty[s], ((i / kStagesF) - 1) & 1, a.status, abort_flag);
      };
      for (int unit = blockIdx.x; unit < n_units && go; unit += gridDim.x) {
        const int u = unit / upe, r0 = (unit - u * upe) * R;
        const int slot = p_slot[u];
        const uint8_t* blob = a.pool + (long long)slot * a.expert_bytes;
        for (int r = r0; r < r0 + R && go; r += P, ++i) {  // phase A: P Wg rows, then the same P Wu rows
          if (i < i_pre) continue;  // issued before griddepcontrol.wait
          const int s = i % kStagesF;
          if (!stage_free(s)) {
            go = false;
            break;
          }
          const uint32_t b = (uint32_t)(P * row_g);
          mbar_expect_tx(&full[s], 2 * b);
          bulk_g2s(ring + (size_t)s * kStageF, blob + r * row_g, b, &full[s]);
          bulk_g2s(ring + (size_t)s * kStageF + b, blob + ((long long)I + r) * row_g, b, &full[s]);
        }
        for (int bx = 0; bx < n_boxes && go; bx += 2, ++i) {  // phase B: two Wd boxes per stage
          const int s = i % kStagesF;
          if (!stage_free(s)) {
            go = false;
            break;
          }
          const int nb = min(2, n_boxes - bx);
          mbar_expect_tx(&full[s], (uint32_t)(nb * kBoxBytes));
          for (int j = 0; j < nb; ++j)
            tma_3d(ring + (size_t)s * kStageF + j * kBoxBytes, &wd_map, r0 * WSZ, (bx + j) * kBoxRows, slot, &full[s]);
        }
      }
      // no copy may still be writing this CTA's shared memory when it exits
      for (int j = i - kStagesF < 0 ? 0 : i - kStagesF; j < i; ++j)
        mbar_wait(&full[j % kStagesF], (j / kStagesF) & 1, a.status);
    }
    return;
  }

  // ---- consumers
  const int ctid = threadIdx.x;  // 0 .. 255
  if (blockIdx.x == 0) {  // y = 0, then the flag that lets every CTA add into it
    const int n4 = T * H / 4;
    for (int i = ctid; i < n4; i += kCons * 32) reinterpret_cast<float4*>(a.y)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    __threadfence();
    cons_sync();
    if (ctid == 0) asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(y_flag), "r"(event) : "memory");
  }
  bool y_ready = blockIdx.x == 0;
  const int sblk_g = H / 128, sblk_d = I / 128;
  const int sbase_d = 2 * (I / 128) * (H / 128);
  int i = 0;
  for (int unit = blockIdx.x; unit < n_units; unit += gridDim.x) {
    const int u = unit / upe, r0 = (unit - u * upe) * R;
    const int row0 = p_off[u];
    const int nrows_all = min(p_off[u + 1] - row0, kMaxT);  // T <= kMaxT rows at most
    const uint8_t* blob = a.pool + (long long)p_slot[u] * a.expert_bytes;
    if constexpr (WT == FT_W_FP8E4M3_B128) {
      // the unit's block scales, read once: its rows lie in one 128-row block of
      // Wg and Wu (one scale per 128-wide K block each) and its Wd columns in one
      // 128-column block (one scale per 128-row block of Wd)
      const int rb = r0 >> 7;
      for (int j = ctid; j < 3 * sblk_g; j += kCons * 32) {
        const int idx = j < sblk_g       ? rb * sblk_g + j
                        : j < 2 * sblk_g ? (I / 128) * sblk_g + rb * sblk_g + (j - sblk_g)
                                         : sbase_d + (j - 2 * sblk_g) * sblk_d + rb;
        s_sc[j] = scale_at(blob, scale_off, idx);
      }
      cons_sync();
    }
    // phase A: h' = w * silu(Wg x) * (Wu x) for the unit's R rows
    const int nch = (int)(row_g / 16);
    for (int r = r0, sidx = 0; r < r0 + R; r += P, ++sidx, ++i) {
      const int s = i % kStagesF;
      const bool ok = acquire(&full[s], (i / kStagesF) & 1, a.status, abort_flag);
      for (int jp = 0; jp < P && ok; ++jp) {
        if ((sidx * P + jp) % kCons != warp) continue;
        const uint4* grow = reinterpret_cast<const uint4*>(ring + (size_t)s * kStageF + jp * row_g);
        const uint4* urow = reinterpret_cast<const uint4*>(ring + (size_t)s * kStageF + (P + jp) * row_g);
        const int rr = r + jp;
        for (int g0 = 0; g0 < nrows_all; g0 += MR) {
        const int nrows = min(nrows_all - g0, MR);
        float wq[MR];
        const uint8_t* xrow[MR];
#pragma unroll
        for (int q = 0; q < MR; ++q) {
          const int row = q < nrows ? p_rows[row0 + g0 + q] : 0;
          wq[q] = q < nrows ? p_w[row] : 0.0f;
          xrow[q] = xs + (size_t)(row / k) * H * act_bytes;
        }
        float ag[MR], au[MR];
#pragma unroll
        for (int q = 0; q < MR; ++q) ag[q] = au[q] = 0.0f;
#pragma unroll
        for (int ci = 0; ci < NCL; ++ci) {
          const int c = ci * 32 + lane;
          if (c >= nch) break;
          float fg[EPC], fu[EPC];
          decode_chunk<WT>(grow[c], fg);
          decode_chunk<WT>(urow[c], fu);
          float sg = 1.0f, su = 1.0f;
          if (WT == FT_W_FP8E4M3_B128) {
            const int cb = (c * EPC) >> 7;
            sg = s_sc[cb];
            su = s_sc[sblk_g + cb];
          }
#pragma unroll
          for (int q = 0; q < MR; ++q) {
            if (q < nrows) {
              float xv[EPC];
              load_act<kF32, EPC>(xrow[q], c * EPC, xv);
              float pg0 = 0.0f, pg1 = 0.0f, pu0 = 0.0f, pu1 = 0.0f;
#pragma unroll
              for (int e = 0; e < EPC; e += 2) {
                pg0 = fmaf(fg[e], xv[e], pg0);
                pu0 = fmaf(fu[e], xv[e], pu0);
                pg1 = fmaf(fg[e + 1], xv[e + 1], pg1);
                pu1 = fmaf(fu[e + 1], xv[e + 1], pu1);
              }
              ag[q] = fmaf(sg, pg0 + pg1, ag[q]);
              au[q] = fmaf(su, pu0 + pu1, au[q]);
            }
          }
        }
#pragma unroll
        for (int q = 0; q < MR; ++q) {
          if (q < nrows) {
            const float g = warp_sum(ag[q]);
            const float v = warp_sum(au[q]);
            if (lane == q) hs[(g0 + q) * R + (rr - r0)] = wq[q] * (g / (1.0f + expf(-g)) * v);
          }
        }
        }
      }
      release(&empty[s]);
    }
    cons_sync();  // h' of the unit is complete
    if (!y_ready) {  // CTA 0 has zeroed y (long done by now): wait, bounded, for its flag
      if (ctid == 0) {
        const unsigned long long t0 = global_ns();
        for (;;) {
          int v;
          asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(y_flag) : "memory");
          if (v == event) break;
          if (*abort_flag || global_ns() - t0 > kWaitLimitNs) {
            if (!*abort_flag && a.status) atomicCAS(a.status, 0, (int)FT_ERR_TIMEOUT);
            *abort_flag = 1;
            break;
          }
        }
      }
      cons_sync();
      y_ready = true;
    }
    // phase B: y[t][c] += sum_i Wd[c][r0 + i] h'[t][i], one output row per thread and box
    for (int bx = 0; bx < n_boxes; bx += 2, ++i) {
      const int s = i % kStagesF;
      const bool ok = acquire(&full[s], (i / kStagesF) & 1, a.status, abort_flag);
      const int nb = ok ? min(2, n_boxes - bx) : 0;
      for (int j = 0; j < nb; ++j) {
        const uint8_t* box = ring + (size_t)s * kStageF + j * kBoxBytes;
        const int c = (bx + j) * kBoxRows + ctid;
        float sc = 1.0f;
        if (WT == FT_W_FP8E4M3_B128) sc = s_sc[2 * sblk_g + (c >> 7)];
        for (int g0 = 0; g0 < nrows_all; g0 += MR) {
        const int nrows = min(nrows_all - g0, MR);
        float acc[MR];
#pragma unroll
        for (int q = 0; q < MR; ++q) acc[q] = 0.0f;
#pragma unroll
        for (int ch = 0; ch < kSlice / 16; ++ch) {
          float f[EPC];
          decode_chunk<WT>(box_get16(box, ctid, ch), f);
#pragma unroll
          for (int q = 0; q < MR; ++q) {
            if (q < nrows) {
              const float* hq = hs + (g0 + q) * R + ch * EPC;
              float p0 = 0.0f, p1 = 0.0f;
#pragma unroll
              for (int e = 0; e < EPC; e += 2) {
                p0 = fmaf(f[e], hq[e], p0);
                p1 = fmaf(f[e + 1], hq[e + 1], p1);
              }
              acc[q] += p0 + p1;
            }
          }
        }
#pragma unroll
        for (int q = 0; q < MR; ++q)
          if (q < nrows) atomicAdd(a.y + (long long)(p_rows[row0 + g0 + q] / k) * H + c, sc * acc[q]);
        }
      }
      release(&empty[s]);
    }
    cons_sync();  // the next unit may overwrite h'
  }

  // ---- copy-engine mode: the last CTA to finish resets the flag and tells the
  // copy thread that this event's slots are no longer read.  With SM pull the
  // CTAs just leave: the flag keeps this launch's event, which the next
  // launch (a later event: ft_moe_forward takes each event once) never waits
  // for, so no count of finished CTAs delays the end of the kernel.
  if (!a.done_host) return;
  cons_sync();
  if (ctid == 0) {
    __threadfence();
    if (atomicAdd(done_ctr, 1u) == gridDim.x - 1) {
      *reinterpret_cast<volatile unsigned*>(done_ctr) = 0u;
      atomicExch(y_flag, 0xffffffffu);
      if (a.done_host) {
        __threadfence_system();
        asm volatile("st.release.sys.global.b32 [%0], %1;" ::"l"(a.done_host + (event % kRing)), "r"(event)
                     : "memory");
      }
    }
  }
}

int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
  }
  return n;
}

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Wd of every slot as a 3D byte tensor: [slot][row c < H][I * wsize bytes],
// boxes of 64 bytes x 256 rows x 1 slot, 64-byte swizzle.
cudaError_t wd_map(CUtensorMap* m, const FfnArgs& a, int wsize) {
  static EncodeTiled enc = nullptr;
  if (!enc) enc = reinterpret_cast<EncodeTiled>(driver_fn("cuTensorMapEncodeTiled"));
  if (!enc) return cudaErrorNotSupported;
  const uint8_t* base = a.pool + 2LL * a.H * a.I * wsize;
  if ((reinterpret_cast<uintptr_t>(base) & 15) || (a.expert_bytes & 15)) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {(cuuint64_t)a.I * wsize, (cuuint64_t)a.H, (cuuint64_t)a.num_slots};
  const cuuint64_t strides[2] = {(cuuint64_t)a.I * wsize, (cuuint64_t)a.expert_bytes};
  const cuuint32_t box[3] = {kSlice, kBoxRows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorNotSupported;
}

template <int WT, int MR, int NCL>
cudaError_t launch_typed(const FfnArgs& a, const Lay& lay, const CUtensorMap& map, cudaStream_t s) {
  static std::mutex mu;
  static std::map<int, int> limit;  // device -> this instance's dynamic shared memory limit so far (only grows)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  {
    std::lock_guard<std::mutex> lk(mu);
    int& lim = limit[dev];
    if (lay.total > lim) {
      e = cudaFuncSetAttribute(ffn_fused_kernel<WT, MR, NCL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               lay.total);
      if (e == cudaSuccess)  // same split as the route and fetch kernels, so a route CTA can share an SM
        e = cudaFuncSetAttribute(ffn_fused_kernel<WT, MR, NCL>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
      if (e != cudaSuccess) return e;
      lim = lay.total;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sm_count());
  cfg.blockDim = dim3(kThreadsF);
  cfg.dynamicSmemBytes = lay.total;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, ffn_fused_kernel<WT, MR, NCL>, map, a);
}

template <int WT>
cudaError_t fused_typed(const FfnArgs& a, cudaStream_t s) {
  constexpr int WSZ = W<WT>::kBytes;
  if (!a.gbar || a.T < 1 || a.T > kMaxT || a.num_slots < 1) return cudaErrorNotSupported;
  const Lay lay(a.H, a.I, a.T, WSZ, WT == FT_W_F32 ? 4 : 2, a.max_unique, a.T * a.k);
  if (!lay.ok(a.H, a.I, WSZ) || lay.total > 200 * 1024) return cudaErrorNotSupported;
  if ((a.H * WSZ) % 16 || (a.T * a.H * (WT == FT_W_F32 ? 4 : 2)) % 16) return cudaErrorNotSupported;
  CUtensorMap map;
  cudaError_t e = wd_map(&map, a, WSZ);
  if (e != cudaSuccess) return e;
  const int nch = a.H * WSZ / 16;  // 16-byte chunks of one Wg/Wu row
  if (nch <= 64)
    return a.T == 1 ? launch_typed<WT, 1, 2>(a, lay, map, s)
                    : launch_typed<WT, 4, 2>(a, lay, map, s);
  if (nch > 256) return cudaErrorNotSupported;
  return a.T == 1 ? launch_typed<WT, 1, 8>(a, lay, map, s)
                  : launch_typed<WT, 4, 8>(a, lay, map, s);
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

}  // namespace ft
