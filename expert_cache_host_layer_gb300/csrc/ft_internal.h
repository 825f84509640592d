// Internal declarations of libft: device-side table/plan layouts and the
// kernel launchers each .cu file provides.  Not part of the C ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "ft.h"

namespace ft {

constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 32;
constexpr int kDecodeMaxTokens = 8;   // T above this takes the grouped-GEMM path
constexpr int kMaxFetchWarps = 4;      // copy warps of the fused decode FFN kernel
constexpr int kDefaultFetchWarps = 2;  // of which take part by default

// Bounds checks of the table and plan indices the kernels dereference, in
// builds made with -DFT_CHECKED: an index out of its range raises
// FT_ERR_CHECKED in the sticky status word and the kernel skips that access
// (no trap).  In other builds the checks compile away.
#ifdef FT_CHECKED
constexpr bool kChecked = true;
#else
constexpr bool kChecked = false;
#endif
__device__ __forceinline__ bool checked_ok(bool in_range, int32_t* status) {
  if (!kChecked || in_range) return true;
  if (status) atomicCAS(status, 0, (int)FT_ERR_CHECKED);
  return false;
}
// __syncthreads after a CTA staged a plan; in checked builds also whether no
// thread found an index out of range in what it staged (and the report).
__device__ __forceinline__ bool plan_sync(int bad, int32_t* status) {
  if (!kChecked) {
    __syncthreads();
    return true;
  }
  const bool ok = !__syncthreads_or(bad);
  if (threadIdx.x == 0) checked_ok(ok, status);
  return ok;
}

// Stats slots in the device counter array.
enum { ST_EVENTS = 0, ST_UNIQUE, ST_HITS, ST_MISSES, ST_EVICT, ST_BYTES, ST_COUNT };

// Plan header words.
enum { PH_EVENT = 0, PH_TOKENS, PH_UNIQUE, PH_MISS, PH_ROWS, PH_STATUS, PH_WORDS = 8 };

// Global slot tables of one cache (device memory, library-owned).
struct Tables {
  int32_t* key_to_slot;  // [L*E]  slot of key l*E+e, -1 = absent
  int32_t* slot_key;     // [C]    key held by the slot, -1 = empty
  int32_t* slot_ts;      // [C]    event of last use, -1 = never
  // The LRU order as an append-only log of (slot, key) entries: every slot
  // has exactly one live entry, and the live entries from head to tail are in
  // ascending (slot_ts, slot) order.  An event tombstones (slot = -1) the
  // entries of its hits and takes its victims from the head, then appends its
  // slots at the tail in slot order, so it touches O(|U|) entries, not C.
  // Positions are 32-bit counters taken modulo log_cap (a power of two); when
  // an event would not fit, the live entries are compacted into the other
  // buffer first.
  int2* log[2];          // [log_cap] ping-pong buffers
  int32_t* pos;          // [C]    counter of each slot's live entry
  uint32_t* head;        // [1]    counter of the first entry not yet passed
  uint32_t* tail;        // [1]    counter one past the last entry
  int32_t* log_cur;      // [1]    which log buffer is current
  int32_t* status;       // [1]    sticky device status (ft_status), 0 = ok
  int32_t* last_nu;      // [1]    |U| of the last event (its slots are the last entries of the order)
  int32_t* event_ctr;    // [1]    event number of the next classification
  int32_t* pin_next;     // [1]    1: the next event pins the last event's slots (0 after create / resize)
  long long* stats;      // [ST_COUNT]
  int32_t num_slots;
  int32_t log_cap;
  int32_t num_keys;      // L*E
};
// Log capacity for C slots: room for the tombstones of many events between
// compactions (a power of two).
inline int32_t log_capacity(long long C) {
  long long q = 4096;
  while (q < 32 * C) q <<= 1;
  return (int32_t)q;
}

// One layer's plan (device memory, library-owned), written by route_classify.
struct Plan {
  int32_t* hdr;            // [PH_WORDS]
  int32_t* unique_expert;  // [E]  ascending
  int32_t* unique_slot;    // [E]
  int32_t* hit;            // [E]
  int32_t* miss_expert;    // [E]  ascending
  int32_t* miss_slot;      // [E]
  int32_t* evicted_key;    // [E]
  int32_t* e2u;            // [E]  expert -> index in U, -1 if not selected
  int32_t* u_count;        // [E]  rows (token, pick) per unique expert
  int32_t* u_offset;       // [E+1] exclusive prefix of u_count
  int32_t* rows_by_u;      // [max_rows] row ids t*k+j grouped by unique expert, ascending within a group
  int32_t* topk_idx;       // [max_rows]
  float* topk_w;           // [max_rows]
};

// Scratch of the route_classify kernel: zero before a launch, left zero after it.
struct RouteScratch {
  uint32_t* bits;    // [kMaxExperts/32] union of the batch's experts
  int32_t* counts;   // [kMaxExperts]    picks per expert
  uint32_t* ticket;  // [1]              CTAs finished
};

// Copy-engine mode: each route_classify appends its miss list to a ring in
// mapped pinned host memory; it fills the fields, then stamps `event` last.
// A library host thread polls the ring; once the FFN of event - 2 has
// finished (the FFN's last CTA writes its event to done_host[e % kRing], also
// mapped pinned memory) it issues the blob copies, then sets
// ready_flags[event % kRing] = event on the copy stream after them; the FFN
// kernels wait for that flag.  kRing bounds how far routing may run ahead of
// the copies (a step graph routes at most one step of L layers ahead).
constexpr int kRing = 128;
struct RingEntry {
  int32_t event;  // stamp: the event number once the entry is complete
  int32_t layer;
  int32_t n_miss;
  int32_t pad;
  int32_t miss_expert[kMaxExperts];
  int32_t miss_slot[kMaxExperts];
};

struct RouteArgs {
  const float* logits;
  int T, E, k, layer;  // the event number and the pin flag live in the tables (device state)
  int32_t* out_idx;  // optional caller outputs
  float* out_w;
  Tables tab;
  Plan plan;
  RouteScratch scr;
  RingEntry* ring;     // device address of the event ring (copy-engine mode), or null
  long long expert_bytes;
  int build_rows;      // 1: the kernel groups rows by expert (small T*k)
};

// Sets the calling thread's ft_last_error() message and returns `s`.
ft_status set_error(ft_status s, const char* fmt, ...);

cudaError_t launch_route_classify(const RouteArgs& a, cudaStream_t s);
// An SM changes its L1/shared-memory split only when it is empty, so kernels
// that run side by side (route, miss pull, FFN) all ask for the largest
// shared-memory split; otherwise a small-split kernel keeps the FFN's CTAs
// (about 150 KB each) off its SMs until it drains.  Called at cache creation.
cudaError_t prefer_max_shared_route();
cudaError_t prefer_max_shared_fetch();
cudaError_t launch_init_tables(Tables tab, int num_keys, cudaStream_t s);

struct PullArgs {
  const int32_t* hdr;
  const int32_t* miss_expert;
  const int32_t* miss_slot;
  int layer, E;
  long long bank_blobs;
  const void* bank;  // device address of the host bank
  void* pool;
  long long expert_bytes;
  int num_slots;
  int32_t* status;   // sticky status word (FT_ERR_CHECKED in checked builds)
};
cudaError_t launch_pull_misses(const PullArgs& a, int ctas, cudaStream_t s);

struct FfnArgs {
  const int32_t* hdr;
  const int32_t* unique_slot;
  const int32_t* hit;        // [n_unique] 1: the expert was in its slot before this event (no copy writes it now)
  const int32_t* u_offset;
  const int32_t* rows_by_u;
  const float* topk_w;
  const void* x;   // [T][H] f32 or bf16
  float* y;        // [T][H] f32
  const uint8_t* pool;
  long long expert_bytes;
  int num_slots;   // slots of the pool (the fused kernel's tensor map of Wd spans them all)
  int H, I, k, T, wdtype;
  int max_unique;  // upper bound of the plan's n_unique (min(T*k, E)), sizes the grid
  float* h;        // [T*k][I] intermediate
  int32_t* status; // sticky status word (bounded waits record FT_ERR_TIMEOUT)
  unsigned* gbar;  // [4] of the fused kernel: [2] finished-CTA count (copy-engine mode; 0 between
                   // launches), [3] the event whose y is zeroed (copy-engine mode: 0xffffffff between
                   // launches; SM pull: the last launch's event); [0], [1] unused
  const int32_t* ready_flags;  // copy-engine mode: wait for ready_flags[e % kRing] == e (e = plan event); or null
  int32_t* done_host;          // copy-engine mode: device address of the mapped [kRing] words where the
                               // FFN stores e at done_host[e % kRing] once it no longer reads its slots; or null
  PullArgs nx;                 // SM-pull mode: the next event's miss fetch, done by the fused kernel's copy
                               // warps while it computes (nx.hdr null: none)
  int fetch_warps;             // how many of the kernel's copy warps take part (1..kMaxFetchWarps)
};
// Copy-engine mode, two-kernel path or T == 0: one thread stores the plan's
// event into done_host after the work before it on the stream.
cudaError_t launch_signal_done(const FfnArgs& a, cudaStream_t s);
// Prefill path (T > kDecodeMaxTokens, bf16 weights): grouped rows, the
// gate/up + SwiGLU grouped GEMM, the down grouped GEMM, the combine.
struct PrefillArgs {
  const int32_t* hdr;
  const int32_t* unique_expert;
  const int32_t* unique_slot;
  const int32_t* u_offset;
  const int32_t* topk_idx;   // [T*k]
  const float* topk_w;       // [T*k]
  int32_t* rows_by_u;        // [T*k] out: rows grouped by unique expert
  int32_t* pos;              // [T*k] out: grouped place of each row
  int32_t* hist;             // [E][group_chunks(T*k)] scratch of the row grouping
  const void* x;             // [T][H] bf16
  void* xp;                  // [T*k][H] bf16 scratch: the x row of each grouped row
  void* h;                   // [T*k][I] bf16 scratch
  void* yp;                  // [T*k][H] fp16 scratch: each row's gate-weighted down projection
  float* y;                  // [T][H] fp32 out
  const uint8_t* pool;
  long long expert_bytes;
  int32_t* status;           // sticky status word (bounded waits record FT_ERR_TIMEOUT)
  int H, I, k, T, E;
  int wdtype;                // FT_W_BF16 or FT_W_FP8E4M3_B128
};
bool prefill_supported(int H, int I, int wdtype, int E);
int group_chunks(long long rows);  // chunks of rows the prefill row grouping counts separately
void prefill_init();               // works out the prefill kernels' grids (call outside stream capture)
// marks (optional): events recorded before and after the gate/up GEMM, then
// before and after the down GEMM.
cudaError_t launch_prefill_ffn(const PrefillArgs& a, int num_slots, cudaStream_t s, int* launches,
                               const cudaEvent_t* marks);
// The two grouped GEMMs of the prefill path on tcgen05 (prefill_tc.cu).
bool prefill_tc_supported(int H, int I);
cudaError_t launch_prefill_gemms(const PrefillArgs& a, int num_slots, cudaStream_t s, const cudaEvent_t* marks);

// Decode path: the gate/up+SwiGLU kernel, then the down+combine kernel.
cudaError_t launch_decode_gateup(const FfnArgs& a, cudaStream_t s);
cudaError_t launch_decode_down(const FfnArgs& a, cudaStream_t s);
// Both in one kernel per layer (decode_fused.cu: units of intermediate rows,
// each CTA adds its units' down projections into y; no grid barrier), launched
// as a programmatic dependent of the previous kernel on the stream;
// cudaErrorNotSupported when the shape does not fit it (the caller then uses
// the two kernels).
cudaError_t launch_decode_ffn_fused(const FfnArgs& a, cudaStream_t s);

struct ResizeArgs {
  Tables old_tab;
  Tables new_tab;  // num_slots = C'
  int num_keys, E;
  int32_t* moves;     // [2*C'] (old, new) pairs
  int32_t* n_moves;   // [1]
  int copy_all;       // 1: pools differ, every survivor moves
};
cudaError_t launch_resize_tables(const ResizeArgs& a, cudaStream_t s, int* launches);
cudaError_t launch_move_blobs(const int32_t* moves, const int32_t* n_moves, int max_moves, const void* src_pool,
                              void* dst_pool, long long expert_bytes, cudaStream_t s);

}  // namespace ft
