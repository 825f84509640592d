// route_classify: one kernel per MoE layer event that does the whole routing
// and cache-decision step with no host sync ("FreeToken: Efficient
// Edge-Native MoE Serving with Bandwidth-Adaptive Execution", design
// paragraph: routing dedup, hit classification and LRU victim selection in one
// GPU kernel, avoiding a per-layer host synchronisation).
//
// Phase 1 (all CTAs): one warp per token computes the top-k experts by logit
// (descending, lower index on ties; NaN ordered as -inf) with k rounds of a
// warp-wide arg-max, and the gates softmax(selected logits).  Each CTA ORs its
// tokens' experts into a shared bit set and counts picks per expert.  With
// more than one CTA, the CTAs merge both into global scratch (one atomic per
// non-zero word/count) and the last CTA to finish (atomic ticket) runs phase
// 2; a single CTA (decode) keeps everything in shared memory.
//
// Phase 2 (one CTA): dedup (the bit set in ascending order is U), hit
// classification against key_to_slot, global-LRU victims, table updates and
// the plan.  The LRU order is an append-only log of (slot, key) entries with
// one live entry per slot, live entries in (last use, slot) order from head to
// tail.  The previous event appended its slots last, so they are the log's
// last |U_{t-1}| entries: the pin rule is "stop before them".  An event
// tombstones its hits' entries, takes the first |M| live entries from the
// head as victims (one warp, a ballot per 32 entries), advances the head past
// dead entries and appends its slots, in slot order, at the tail: O(|U|) work
// plus the tombstones it passes, instead of a pass over all C slots.
#include <cfloat>
#include <climits>

#include "ft_internal.h"

namespace ft {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// Exclusive block-wide prefix sum of one int per thread; `total` gets the sum.
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

// key_to_slot[key]; in checked builds a slot out of range, or one whose
// slot_key is not the key, is reported and read as absent.
__device__ __forceinline__ int checked_slot(const Tables& t, int key) {
  const int s = t.key_to_slot[key];
  if (!kChecked || s == -1) return s;
  return checked_ok(s >= 0 && s < t.num_slots && t.slot_key[s] == key, t.status) ? s : -1;
}

template <int PL>  // logits per lane: E <= 32 * PL
__global__ void __launch_bounds__(kThreads) route_classify_kernel(RouteArgs a) {
  __shared__ uint32_t s_bits[kMaxExperts / 32];
  __shared__ int s_cnt[kMaxExperts];
  __shared__ int s_warp[kWarps];
  __shared__ int s_wpre[33];
  __shared__ int s_uexp[kMaxExperts];
  __shared__ int s_uslot[kMaxExperts];
  __shared__ int s_mrank[kMaxExperts];  // miss rank of each unique expert, -1 for hits
  __shared__ int s_missexp[kMaxExperts];
  __shared__ int s_victim[kMaxExperts];
  __shared__ int s_evict[kMaxExperts];
  __shared__ int s_uoff[kMaxExperts];
  __shared__ int s_rowu[kMaxExperts];
  __shared__ int s_k2s[kMaxExperts];  // key_to_slot of this layer's experts
  __shared__ int s_flag;
  __shared__ uint32_t s_head;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = a.E, k = a.k, T = a.T;
  const int nwords = (E + 31) >> 5;
  const bool single = gridDim.x == 1;

  for (int i = tid; i < nwords; i += kThreads) s_bits[i] = 0u;
  for (int i = tid; i < E; i += kThreads) s_cnt[i] = 0;
  // A single CTA runs phase 2 itself: start its table reads now so they
  // overlap the top-k work (the multi-CTA tail reads them after the ticket).
  const int layer = a.layer;
  int cur = 0, event = 0, n_prev = 0;
  uint32_t head = 0, tail = 0;
  if (single) {
    cur = *a.tab.log_cur;
    event = *a.tab.event_ctr;
    n_prev = *a.tab.pin_next ? *a.tab.last_nu : 0;
    head = *a.tab.head;
    tail = *a.tab.tail;
    for (int e = tid; e < E; e += kThreads) s_k2s[e] = checked_slot(a.tab, layer * E + e);
  }
  __syncthreads();

  // ---------------- phase 1: top-k + gates, one warp per token -------------
  for (int t = blockIdx.x * kWarps + warp; t < T; t += gridDim.x * kWarps) {
    const float* row = a.logits + (long long)t * E;
    float v[PL];
#pragma unroll
    for (int q = 0; q < PL; ++q) {
      const int e = q * 32 + lane;
      float x = e < E ? __ldg(row + e) : -INFINITY;
      v[q] = (x != x) ? -INFINITY : x;  // NaN ordered as -inf
    }
    uint32_t taken = 0u;
    float my_v = -INFINITY;
    int my_i = 0;
    for (int j = 0; j < k; ++j) {
      float bv = -INFINITY;
      int bi = INT_MAX;
#pragma unroll
      for (int q = 0; q < PL; ++q) {
        const int e = q * 32 + lane;
        if (e < E && !((taken >> q) & 1u) && better(v[q], e, bv, bi)) {
          bv = v[q];
          bi = e;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (better(ov, oi, bv, bi)) {
          bv = ov;
          bi = oi;
        }
      }
      if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
      if (lane == j) {
        my_v = bv;
        my_i = bi;
      }
    }
    const float m = __shfl_sync(0xffffffffu, my_v, 0);
    float ex = lane < k ? expf(my_v - m) : 0.0f;
    float sum = ex;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane < k) {
      const float w = ex / sum;
      const long long r = (long long)t * k + lane;
      a.plan.topk_idx[r] = my_i;
      a.plan.topk_w[r] = w;
      if (a.out_idx) a.out_idx[r] = my_i;
      if (a.out_w) a.out_w[r] = w;
      atomicOr(&s_bits[my_i >> 5], 1u << (my_i & 31));
      atomicAdd(&s_cnt[my_i], 1);
    }
  }
  __syncthreads();
  if (!single) {  // merge into global scratch; the last CTA continues
    for (int i = tid; i < nwords; i += kThreads)
      if (s_bits[i]) atomicOr(&a.scr.bits[i], s_bits[i]);
    for (int i = tid; i < E; i += kThreads)
      if (s_cnt[i]) atomicAdd(&a.scr.counts[i], s_cnt[i]);
    __threadfence();
    __syncthreads();
    if (tid == 0) s_flag = (atomicAdd(a.scr.ticket, 1u) == gridDim.x - 1);
    __syncthreads();
    if (!s_flag) return;
    __threadfence();
    for (int i = tid; i < nwords; i += kThreads) s_bits[i] = __ldcg(&a.scr.bits[i]);
    for (int i = tid; i < E; i += kThreads) s_cnt[i] = __ldcg(&a.scr.counts[i]);
    __syncthreads();
  }

  // ---------------- phase 2 (one CTA): dedup, classify, victims ------------
  if (!single) {
    cur = *a.tab.log_cur;
    event = *a.tab.event_ctr;
    n_prev = *a.tab.pin_next ? *a.tab.last_nu : 0;
    head = *a.tab.head;
    tail = *a.tab.tail;
    for (int e = tid; e < E; e += kThreads) s_k2s[e] = checked_slot(a.tab, layer * E + e);
  }
  if (warp == 0) {
    int c = lane < nwords ? __popc(s_bits[lane]) : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, c, o);
      if (lane >= o) c += y;
    }
    s_wpre[lane + 1] = c;
    if (lane == 0) s_wpre[0] = 0;
  }
  __syncthreads();
  const int n_u = s_wpre[nwords];
  for (int e = tid; e < E; e += kThreads) {
    const int w = e >> 5, b = e & 31;
    if ((s_bits[w] >> b) & 1u) {
      const int u = s_wpre[w] + __popc(s_bits[w] & ((1u << b) - 1u));
      s_uexp[u] = e;
      a.plan.e2u[e] = u;
    } else {
      a.plan.e2u[e] = -1;
    }
  }
  __syncthreads();

  // hit classification and miss ranks (ascending expert order)
  int carry = 0;
  for (int base = 0; base < n_u; base += kThreads) {
    const int u = base + tid;
    int is_miss = 0;
    if (u < n_u) {
      const int s = s_k2s[s_uexp[u]];
      s_uslot[u] = s;
      is_miss = s < 0;
    }
    int tot;
    const int r = block_excl_scan(is_miss, s_warp, tot);
    if (u < n_u) {
      s_mrank[u] = is_miss ? carry + r : -1;
      if (is_miss) s_missexp[carry + r] = s_uexp[u];
    }
    carry += tot;
  }
  const int n_miss = carry;

  // the LRU log: compact it first if this event's entries would not fit
  const uint32_t Q = (uint32_t)a.tab.log_cap, qmask = Q - 1;
  if (tail - head + (uint32_t)n_u > Q) {
    const int2* src = a.tab.log[cur];
    int2* dst = a.tab.log[cur ^ 1];
    int kept = 0;
    for (uint32_t base = head; base != tail;) {
      const uint32_t n = min((uint32_t)kThreads, tail - base);
      int2 e = make_int2(-1, -1);
      if ((uint32_t)tid < n) e = src[(base + tid) & qmask];
      const int live = (uint32_t)tid < n && e.x >= 0;
      int tot;
      const int r = block_excl_scan(live, s_warp, tot);
      if (live) {
        dst[kept + r] = e;
        a.tab.pos[e.x] = kept + r;
      }
      kept += tot;
      base += n;
    }
    // the previous event's entries stay the last ones (compaction keeps the order)
    cur ^= 1;
    head = 0;
    tail = (uint32_t)kept;
    __syncthreads();
  }
  int2* lg = a.tab.log[cur];
  // tombstone the hits' entries
  for (int u = tid; u < n_u; u += kThreads)
    if (s_mrank[u] < 0) lg[(uint32_t)a.tab.pos[s_uslot[u]] & qmask].x = -1;
  __syncthreads();
  // victims: the first n_miss live entries from the head, stopping before the
  // previous event's entries (pinned); then the head passes the dead entries
  const uint32_t pin_start = tail - (uint32_t)n_prev;
  if (warp == 0) {
    int found = 0;
    uint32_t p = head;
    while (found < n_miss && p != pin_start) {
      const uint32_t n = min(32u, pin_start - p);
      int2 e = (uint32_t)lane < n ? lg[(p + lane) & qmask] : make_int2(-1, -1);
      if (kChecked && e.x >= 0 && !checked_ok(e.x < a.tab.num_slots && e.y >= -1 && e.y < a.tab.num_keys, a.tab.status))
        e = make_int2(-1, -1);  // a corrupt entry is reported and never taken
      const bool live = (uint32_t)lane < n && e.x >= 0;
      const unsigned m = __ballot_sync(0xffffffffu, live);
      const int r = found + __popc(m & ((1u << lane) - 1u));
      if (live && r < n_miss) {
        s_victim[r] = e.x;
        s_evict[r] = e.y;
        lg[(p + lane) & qmask].x = -1;
      }
      found = min(n_miss, found + __popc(m));
      p += n;
    }
    if (lane == 0) s_flag = found;
    __syncwarp();
    // head: first live entry at or after the old head (bounded by the tail)
    uint32_t h = head;
    while (h != tail) {
      const uint32_t n = min(32u, tail - h);
      const bool live = (uint32_t)lane < n && lg[(h + lane) & qmask].x >= 0;
      const unsigned m = __ballot_sync(0xffffffffu, live);
      if (m) {
        h += __ffs(m) - 1;
        break;
      }
      h += n;
    }
    if (lane == 0) s_head = h;
  }
  __syncthreads();
  const bool capacity_ok = s_flag >= n_miss;

  if (!capacity_ok) {  // pool too small for this event: put the log back and leave the tables as they are
    for (int u = tid; u < n_u; u += kThreads)
      if (s_mrank[u] < 0) lg[(uint32_t)a.tab.pos[s_uslot[u]] & qmask].x = s_uslot[u];
    for (int i = tid; i < s_flag; i += kThreads) lg[(uint32_t)a.tab.pos[s_victim[i]] & qmask].x = s_victim[i];
    if (tid == 0) {
      atomicCAS(a.tab.status, 0, (int)FT_ERR_CAPACITY);
      a.plan.hdr[PH_EVENT] = event;
      a.plan.hdr[PH_STATUS] = (int)FT_ERR_CAPACITY;
      a.plan.hdr[PH_MISS] = 0;
      a.plan.hdr[PH_UNIQUE] = 0;
      *a.tab.last_nu = 0;
      *a.tab.event_ctr = event + 1;
      *a.tab.pin_next = 1;
      *a.tab.log_cur = cur;
      *a.tab.head = head;
      *a.tab.tail = tail;
      if (a.ring) {
        RingEntry* r = a.ring + (event % kRing);
        r->layer = layer;
        r->n_miss = 0;
      }
    }
  } else {
    // the event's slots (hits and victims) go to the end of the log in slot order
    for (int u = tid; u < n_u; u += kThreads)
      if (s_mrank[u] >= 0) s_uslot[u] = s_victim[s_mrank[u]];
    __syncthreads();
    for (int u = tid; u < n_u; u += kThreads) {
      const int s = s_uslot[u];
      int rank = 0;
      for (int q = 0; q < n_u; ++q) rank += s_uslot[q] < s;
      const uint32_t at = tail + (uint32_t)rank;
      lg[at & qmask] = make_int2(s, layer * E + s_uexp[u]);
      a.tab.pos[s] = (int32_t)at;
      a.tab.slot_ts[s] = event;
      a.plan.unique_expert[u] = s_uexp[u];
      a.plan.unique_slot[u] = s;
      a.plan.hit[u] = s_mrank[u] < 0;
    }
    // table updates: victims lose their key, misses take their victim
    int n_evict = 0;
    for (int i = tid; i < n_miss; i += kThreads) {
      const int s = s_victim[i];
      const int old = s_evict[i];
      a.plan.evicted_key[i] = old;
      if (old >= 0) {
        a.tab.key_to_slot[old] = -1;
        ++n_evict;
      }
      const int key = layer * E + s_missexp[i];
      a.tab.key_to_slot[key] = s;
      a.tab.slot_key[s] = key;
      a.plan.miss_expert[i] = s_missexp[i];
      a.plan.miss_slot[i] = s;
      if (a.ring) {
        RingEntry* r = a.ring + (event % kRing);
        r->miss_expert[i] = s_missexp[i];
        r->miss_slot[i] = s;
      }
    }
    // rows per unique expert and their offsets
    int off = 0;
    for (int base = 0; base < n_u; base += kThreads) {
      const int u = base + tid;
      const int c = u < n_u ? s_cnt[s_uexp[u]] : 0;
      int tot;
      const int r = block_excl_scan(c, s_warp, tot);
      if (u < n_u) {
        a.plan.u_count[u] = c;
        a.plan.u_offset[u] = off + r;
        s_uoff[u] = off + r;
      }
      off += tot;
    }
    if (tid == 0) a.plan.u_offset[n_u] = off;
    if (a.build_rows) {  // small T*k (<= kMaxExperts): rank each row among the rows of its expert
      const int rows = T * k;
      for (int r = tid; r < rows; r += kThreads) {
        const int e = single ? a.plan.topk_idx[r] : __ldcg(&a.plan.topk_idx[r]);
        s_rowu[r] = s_wpre[e >> 5] + __popc(s_bits[e >> 5] & ((1u << (e & 31)) - 1u));
      }
      __syncthreads();
      for (int r = tid; r < rows; r += kThreads) {
        const int u = s_rowu[r];
        int before = 0;
        for (int q = 0; q < r; ++q) before += s_rowu[q] == u;
        a.plan.rows_by_u[s_uoff[u] + before] = r;
      }
    }
    int tot_evict;
    block_excl_scan(n_evict, s_warp, tot_evict);
    if (tid == 0) {
      a.plan.hdr[PH_EVENT] = event;
      a.plan.hdr[PH_TOKENS] = T;
      a.plan.hdr[PH_UNIQUE] = n_u;
      a.plan.hdr[PH_MISS] = n_miss;
      a.plan.hdr[PH_ROWS] = T * k;
      a.plan.hdr[PH_STATUS] = 0;
      long long* st = a.tab.stats;
      st[ST_EVENTS] += 1;
      st[ST_UNIQUE] += n_u;
      st[ST_HITS] += n_u - n_miss;
      st[ST_MISSES] += n_miss;
      st[ST_EVICT] += tot_evict;
      st[ST_BYTES] += (long long)n_miss * a.expert_bytes;
      if (a.ring) {
        RingEntry* r = a.ring + (event % kRing);
        r->layer = layer;
        r->n_miss = n_miss;
      }
      *a.tab.last_nu = n_u;
      *a.tab.event_ctr = event + 1;
      *a.tab.pin_next = 1;
      *a.tab.log_cur = cur;
      *a.tab.head = s_head;
      *a.tab.tail = tail + (uint32_t)n_u;
    }
  }
  if (a.ring) {  // publish the entry: every field first, then the stamp (release, system scope)
    __threadfence_system();
    __syncthreads();
    if (tid == 0)
      asm volatile("st.release.sys.global.b32 [%0], %1;" ::"l"(&a.ring[event % kRing].event), "r"(event) : "memory");
  }
  if (!single) {  // leave the scratch zeroed for the next launch
    for (int i = tid; i < nwords; i += kThreads) a.scr.bits[i] = 0u;
    for (int i = tid; i < E; i += kThreads) a.scr.counts[i] = 0;
    if (tid == 0) *a.scr.ticket = 0u;
  }
}

__global__ void init_tables_kernel(Tables tab, int num_keys) {
  const int stride = gridDim.x * blockDim.x;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < num_keys; i += stride) tab.key_to_slot[i] = -1;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < tab.num_slots; i += stride) {
    tab.slot_key[i] = -1;
    tab.slot_ts[i] = -1;
    tab.log[0][i] = make_int2(i, -1);  // all slots empty: (ts = -1, slot) order is slot order
    tab.pos[i] = i;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    *tab.log_cur = 0;
    *tab.head = 0;
    *tab.tail = (uint32_t)tab.num_slots;
    *tab.status = 0;
    *tab.last_nu = 0;
    *tab.event_ctr = 0;
    *tab.pin_next = 0;
    for (int i = 0; i < ST_COUNT; ++i) tab.stats[i] = 0;
  }
}

}  // namespace

cudaError_t prefer_max_shared_route() {
  const void* fns[] = {reinterpret_cast<const void*>(route_classify_kernel<1>),
                       reinterpret_cast<const void*>(route_classify_kernel<2>),
                       reinterpret_cast<const void*>(route_classify_kernel<4>),
                       reinterpret_cast<const void*>(route_classify_kernel<8>),
                       reinterpret_cast<const void*>(route_classify_kernel<16>),
                       reinterpret_cast<const void*>(route_classify_kernel<32>)};
  for (const void* f : fns) {
    const cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout,
                                               cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_route_classify(const RouteArgs& a, cudaStream_t s) {
  const int warps_needed = (a.T + kWarps - 1) / kWarps;
  int grid = warps_needed < 1 ? 1 : warps_needed;
  if (grid > 4 * 152) grid = 4 * 152;
  const int pl = (a.E + 31) / 32;
  if (pl <= 1)
    route_classify_kernel<1><<<grid, kThreads, 0, s>>>(a);
  else if (pl <= 2)
    route_classify_kernel<2><<<grid, kThreads, 0, s>>>(a);
  else if (pl <= 4)
    route_classify_kernel<4><<<grid, kThreads, 0, s>>>(a);
  else if (pl <= 8)
    route_classify_kernel<8><<<grid, kThreads, 0, s>>>(a);
  else if (pl <= 16)
    route_classify_kernel<16><<<grid, kThreads, 0, s>>>(a);
  else
    route_classify_kernel<32><<<grid, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_init_tables(Tables tab, int num_keys, cudaStream_t s) {
  int n = num_keys > tab.num_slots ? num_keys : tab.num_slots;
  int grid = (n + 255) / 256;
  if (grid > 1024) grid = 1024;
  if (grid < 1) grid = 1;
  init_tables_kernel<<<grid, 256, 0, s>>>(tab, num_keys);
  return cudaGetLastError();
}

}  // namespace ft
