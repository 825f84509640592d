// Cache resize at a scheduler safe point ("FreeToken: Efficient Edge-Native
// MoE Serving ...", design paragraph: when the VRAM budget changes the cache
// is rebuilt at a safe point without restarting the engine).
//
// resize_tables (one CTA): walk the live entries of the LRU log (ascending
// (last use, slot)); drop the first n_occupied - C' occupied ones; survivors
// below C' stay put, survivors at or above C' take the lowest free slots below
// C' in ascending old-slot order.  Writes the new slot tables and the move
// list.  rank_order: rebuilds the log of the new slots, compact, by ranking
// each slot's (last use, slot) key.  move_blobs: copies the moved expert blobs.
#include "ft_internal.h"

namespace ft {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ int block_excl_scan(int v, int* s_warp, int& total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[w] = x;
  __syncthreads();
  if (w == 0) {
    int t = lane < kWarps ? s_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    if (lane < kWarps) s_warp[lane] = t;
  }
  __syncthreads();
  const int before = w > 0 ? s_warp[w - 1] : 0;
  total = s_warp[kWarps - 1];
  __syncthreads();
  return before + x - v;
}

__global__ void __launch_bounds__(kThreads) resize_tables_kernel(ResizeArgs a) {
  __shared__ int s_warp[kWarps];
  const int tid = threadIdx.x;
  const int C = a.old_tab.num_slots, Cn = a.new_tab.num_slots;
  const int cur = *a.old_tab.log_cur;
  const int2* lg = a.old_tab.log[cur];
  const uint32_t qmask = (uint32_t)a.old_tab.log_cap - 1;
  const uint32_t head = *a.old_tab.head, tail = *a.old_tab.tail;
  int32_t* keep = reinterpret_cast<int32_t*>(a.old_tab.log[cur ^ 1]);  // scratch: 1 = survives
  int32_t* free_list = reinterpret_cast<int32_t*>(a.new_tab.log[1]);   // scratch: free slots below C'

  if (kChecked) {  // every slot gets its keep flag from its live log entry; a corrupt log must not leave stale ones
    for (int s = tid; s < C; s += kThreads) keep[s] = 0;
    __syncthreads();
  }
  // occupied count
  int occ_local = 0;
  for (int s = tid; s < C; s += kThreads) occ_local += a.old_tab.slot_key[s] >= 0;
  int n_occ;
  block_excl_scan(occ_local, s_warp, n_occ);
  const int n_drop = n_occ > Cn ? n_occ - Cn : 0;

  // drop the first n_drop occupied live entries of the LRU log
  int carry = 0;
  for (uint32_t base = head; base != tail;) {
    const uint32_t n = min((uint32_t)kThreads, tail - base);
    int s = -1, occ = 0;
    if ((uint32_t)tid < n) {
      s = lg[(base + tid) & qmask].x;
      if (s >= 0 && !checked_ok(s < C && a.old_tab.slot_key[s] < a.old_tab.num_keys, a.old_tab.status)) s = -1;
      occ = s >= 0 && a.old_tab.slot_key[s] >= 0;
    }
    int tot;
    const int r = block_excl_scan(occ, s_warp, tot);
    if (s >= 0) {
      const bool drop = occ && carry + r < n_drop;
      keep[s] = occ && !drop;
      if (drop) a.old_tab.key_to_slot[a.old_tab.slot_key[s]] = -1;
    }
    carry += tot;
    base += n;
  }
  __syncthreads();

  // free slots below C' (not a staying survivor), ascending
  int nfree = 0;
  for (int base = 0; base < Cn; base += kThreads) {
    const int s = base + tid;
    const int f = s < Cn && !(s < C && keep[s]);
    int tot;
    const int r = block_excl_scan(f, s_warp, tot);
    if (f) free_list[nfree + r] = s;
    nfree += tot;
  }
  // empty new tables
  for (int s = tid; s < Cn; s += kThreads) {
    a.new_tab.slot_key[s] = -1;
    a.new_tab.slot_ts[s] = -1;
  }
  __syncthreads();
  // staying survivors
  int n_moves = 0;
  for (int base = 0; base < (C < Cn ? C : Cn); base += kThreads) {
    const int s = base + tid;
    const int stay = s < C && s < Cn && keep[s];
    if (stay) {
      a.new_tab.slot_key[s] = a.old_tab.slot_key[s];
      a.new_tab.slot_ts[s] = a.old_tab.slot_ts[s];
    }
    int tot;
    const int r = block_excl_scan(stay && a.copy_all, s_warp, tot);
    if (stay && a.copy_all) {
      a.moves[2 * (n_moves + r)] = s;
      a.moves[2 * (n_moves + r) + 1] = s;
    }
    n_moves += tot;
  }
  // movers: survivors at or above C', ascending, to the lowest free slots
  int n_movers = 0;
  for (int base = Cn; base < C; base += kThreads) {
    const int s = base + tid;
    const int mv = s < C && keep[s];
    int tot;
    const int r = block_excl_scan(mv, s_warp, tot);
    if (mv && checked_ok(n_movers + r < nfree, a.old_tab.status)) {
      const int d = free_list[n_movers + r];
      const int key = a.old_tab.slot_key[s];
      a.new_tab.slot_key[d] = key;
      a.new_tab.slot_ts[d] = a.old_tab.slot_ts[s];
      a.old_tab.key_to_slot[key] = d;
      a.moves[2 * (n_moves + r)] = s;
      a.moves[2 * (n_moves + r) + 1] = d;
    }
    n_movers += tot;
    n_moves += tot;
  }
  if (tid == 0) {
    *a.n_moves = n_moves;
    *a.new_tab.log_cur = 0;
    *a.new_tab.head = 0;
    *a.new_tab.tail = (uint32_t)Cn;
    *a.new_tab.status = *a.old_tab.status;
    *a.new_tab.last_nu = 0;
    *a.new_tab.event_ctr = *a.old_tab.event_ctr;
    *a.new_tab.pin_next = 0;  // the safe point: nothing of the last event is still being read
    for (int i = 0; i < ST_COUNT; ++i) a.new_tab.stats[i] = a.old_tab.stats[i];
    a.new_tab.stats[ST_EVICT] += n_drop;
  }
}

// log[rank(s)] = (s, key of s), pos[s] = rank(s), with rank by (slot_ts, slot)
// ascending over the new slots: the compact log of the new tables.
__global__ void rank_order_kernel(Tables tab) {
  __shared__ int s_ts[1024];
  const int C = tab.num_slots;
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  const int my = s < C ? tab.slot_ts[s] : 0;
  int rank = 0;
  for (int base = 0; base < C; base += 1024) {
    __syncthreads();
    for (int i = threadIdx.x; i < 1024; i += blockDim.x) s_ts[i] = base + i < C ? tab.slot_ts[base + i] : 0;
    __syncthreads();
    const int n = min(1024, C - base);
    if (s < C)
      for (int i = 0; i < n; ++i) {
        const int o = s_ts[i];
        rank += o < my || (o == my && base + i < s);
      }
  }
  if (s < C) {
    tab.log[0][rank] = make_int2(s, tab.slot_key[s]);
    tab.pos[s] = rank;
  }
}

__global__ void move_blobs_kernel(const int32_t* moves, const int32_t* n_moves_p, const uint4* src, uint4* dst,
                                  long long eb16) {
  const int n_moves = *n_moves_p;
  const long long chunk = 4096;  // 64 KB per item
  const long long per_blob = (eb16 + chunk - 1) / chunk;
  for (long long it = blockIdx.x; it < (long long)n_moves * per_blob; it += gridDim.x) {
    const int m = (int)(it / per_blob);
    const long long c = it - m * per_blob;
    const long long from = moves[2 * m], to = moves[2 * m + 1];
    const long long n = min(chunk, eb16 - c * chunk);
    const uint4* s = src + from * eb16 + c * chunk;
    uint4* d = dst + to * eb16 + c * chunk;
    for (long long i = threadIdx.x; i < n; i += blockDim.x) d[i] = s[i];
  }
}

}  // namespace

cudaError_t launch_resize_tables(const ResizeArgs& a, cudaStream_t s, int* launches) {
  resize_tables_kernel<<<1, kThreads, 0, s>>>(a);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  ++*launches;
  const int Cn = a.new_tab.num_slots;
  rank_order_kernel<<<(Cn + 255) / 256, 256, 0, s>>>(a.new_tab);
  err = cudaGetLastError();
  if (err == cudaSuccess) ++*launches;
  return err;
}

cudaError_t launch_move_blobs(const int32_t* moves, const int32_t* n_moves, int max_moves, const void* src_pool,
                              void* dst_pool, long long expert_bytes, cudaStream_t s) {
  if (max_moves <= 0) return cudaSuccess;
  move_blobs_kernel<<<152 * 4, 256, 0, s>>>(moves, n_moves, static_cast<const uint4*>(src_pool),
                                            static_cast<uint4*>(dst_pool), expert_bytes >> 4);
  return cudaGetLastError();
}

}  // namespace ft
