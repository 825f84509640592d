// Host side of libft: the C ABI declared in include/ft.h.
//
// One ft_cache owns the device slot tables, one plan per layer, the routing
// scratch, (copy-engine mode) a mapped pinned ring of the events' miss lists, the copy
// stream(s) and the per-layer events that order the pipeline:
//
//   compute stream:  route(l+1) -> [cls(l+1)] ... wait(ready(l)) -> FFN(l)
//   copy stream:     wait(cls(l+1)) -> miss copies of l+1 -> [ready(l+1)]
//
// so the misses of layer l+1 stream in while layer l computes ("FreeToken:
// Efficient Edge-Native MoE Serving ...", ablation paragraph: double
// buffering).  In copy-engine mode the route kernel appends each event's miss
// list to a ring in mapped host memory; a library thread polls the ring,
// issues one cudaMemcpyAsync per miss on the copy stream and then a 4-byte
// copy that sets the event's ready flag in device memory; the FFN kernel waits
// (bounded) for that flag.  No host synchronisation sits between the GPU
// work, so a whole step can be captured in a CUDA graph in either mode.  In
// SM-pull mode a kernel on the copy stream reads the device plan itself.
#include <algorithm>
#include <atomic>
#include <climits>
#include <condition_variable>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <chrono>
#include <map>
#include <mutex>
#include <string>
#include <thread>
#include <vector>

#include "ft_internal.h"
#include <nvtx3/nvToolsExt.h>

using namespace ft;

namespace {

thread_local std::string g_last_error;

ft_status fail(ft_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

#define CU(call)                                                                                  \
  do {                                                                                            \
    cudaError_t e_ = (call);                                                                      \
    if (e_ != cudaSuccess)                                                                        \
      return fail(e_ == cudaErrorMemoryAllocation ? FT_ERR_OOM : FT_ERR_CUDA, "%s: %s (%s:%d)", #call, \
                  cudaGetErrorString(e_), __FILE__, __LINE__);                                    \
  } while (0)

size_t blob_bytes(int H, int I, int wdtype) {
  if (H <= 0 || I <= 0) return 0;
  const size_t n = 3ull * H * I;
  switch (wdtype) {
    case FT_W_F32: return (H % 4 || I % 4) ? 0 : 4 * n;
    case FT_W_BF16: return (H % 8 || I % 8) ? 0 : 2 * n;
    case FT_W_FP8E4M3_B128: return (H % 128 || I % 128) ? 0 : n + 2ull * 3 * (H / 128) * (I / 128);
    default: return 0;
  }
}

// Event-pair timer for one phase.  Pairs are folded into the total when the
// pool fills, starting with the oldest (long finished) half.
struct PhaseTimer {
  std::vector<cudaEvent_t> ev;  // 2 per pair
  int used = 0;
  double total_ms = 0.0;
  long long n = 0;
  static constexpr int kPairs = 2048;
  ~PhaseTimer() {
    for (auto e : ev) cudaEventDestroy(e);
  }
  bool ensure() {
    if (!ev.empty()) return true;
    ev.resize(2 * kPairs);
    for (auto& e : ev)
      if (cudaEventCreate(&e) != cudaSuccess) return false;
    return true;
  }
  void fold(int pairs) {
    for (int i = 0; i < pairs; ++i) {
      float ms = 0.0f;
      cudaEventSynchronize(ev[2 * i + 1]);
      if (cudaEventElapsedTime(&ms, ev[2 * i], ev[2 * i + 1]) == cudaSuccess) {
        total_ms += ms;
        ++n;
      }
    }
    // move the unfolded pairs to the front
    for (int i = pairs; i < used; ++i) {
      std::swap(ev[2 * (i - pairs)], ev[2 * i]);
      std::swap(ev[2 * (i - pairs) + 1], ev[2 * i + 1]);
    }
    used -= pairs;
  }
  cudaEvent_t begin(cudaStream_t s) {
    if (!ensure()) return nullptr;
    if (used == kPairs) fold(kPairs / 2);
    cudaEvent_t e = ev[2 * used];
    cudaEventRecord(e, s);
    return e;
  }
  void end(cudaStream_t s) {
    cudaEventRecord(ev[2 * used + 1], s);
    ++used;
  }
  // The next pair, for a caller that records both events itself.
  bool reserve(cudaEvent_t* b, cudaEvent_t* e) {
    if (!ensure()) return false;
    if (used == kPairs) fold(kPairs / 2);
    *b = ev[2 * used];
    *e = ev[2 * used + 1];
    ++used;
    return true;
  }
  void collect() { fold(used); }
  void reset() {
    collect();
    total_ms = 0.0;
    n = 0;
  }
};

enum { PHASE_ROUTE = 0, PHASE_FETCH, PHASE_FFN, PHASE_GEMM1, PHASE_GEMM2, PHASE_COUNT };

}  // namespace

ft_status ft::set_error(ft_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

struct ft_cache {
  // configuration
  ft_cache_config cfg{};
  int L = 0, E = 0, k = 0, H = 0, I = 0, wdtype = 0, max_tokens = 0;
  size_t eb = 0;
  int device = 0;
  // memory
  void* pool = nullptr;
  int64_t C = 0;
  const uint8_t* bank_host = nullptr;
  const void* bank_dev = nullptr;
  bool registered_bank = false;
  Tables tab{};
  std::vector<Plan> plans;
  void* plan_mem = nullptr;
  RouteScratch scr{};
  void* scr_mem = nullptr;
  RingEntry* ring_host = nullptr;     // copy-engine mode: mapped pinned [kRing]
  RingEntry* ring_dev = nullptr;
  int32_t* ready_flags = nullptr;     // device [kRing], set on the copy stream after an event's copies
  int32_t* flag_src = nullptr;        // pinned host [kRing], sources of those 4-byte copies
  int32_t* done_host = nullptr;       // mapped pinned [kRing]: done_host[e % kRing] = e once FFN(e) is done
  int32_t* done_dev = nullptr;        // its device address
  int32_t* counter_host = nullptr;    // pinned host word for reading the device event counter
  float* h_buf = nullptr;             // decode intermediate [max_rows][I]
  // prefill (T > kDecodeMaxTokens): bf16 h [rows][I], fp32 per-row outputs
  // [rows][H], grouped place of each row; allocated only when max_tokens > 8
  void* pf_h = nullptr;
  void* pf_xp = nullptr;              // bf16 x rows in grouped order [rows][H]
  void* pf_yp = nullptr;
  int32_t* pf_pos = nullptr;
  int32_t* pf_hist = nullptr;          // [E][chunks of rows]: the row grouping's counts
  unsigned* gbar = nullptr;           // grid-barrier words of the fused FFN kernel
  bool fused_ok = true;               // false once the fused FFN kernel reported it cannot run
  // streams and events
  cudaStream_t compute = nullptr;
  cudaStream_t route = nullptr;        // route_classify kernels (off the FFN's critical path)
  cudaEvent_t route_join = nullptr;    // compute -> route ordering at each ft_route_classify
  cudaEvent_t slots_free = nullptr;    // compute -> copy ordering when routing runs ahead
  // copy-engine mode: end of each of the last two step-graph launches; a third
  // launch first waits (polling) for the oldest, so the host never queues so
  // much work that a launch call blocks while an FFN waits for the copy thread
  cudaEvent_t inflight[2] = {nullptr, nullptr};
  long long graph_launches = 0;
  // true: routing waits for all compute-stream work (the API's rule); false
  // inside an SM-pull step graph, where every layer's logits are ready at the
  // step's start and only the miss fetch has to wait for the FFN of event t-2
  bool route_follows_compute = true;
  // SM-pull mode: the layer whose fetch was requested but not yet enqueued.
  // The next ft_moe_forward of another layer runs it inside its fused kernel;
  // anything else that needs it first launches it on its own (flush_fetch).
  int pending_fetch = -1;
  cudaStream_t copy[2] = {nullptr, nullptr};
  int ncopy = 1;
  cudaEvent_t copy_join = nullptr;
  std::vector<cudaEvent_t> cls_ev, ready_ev;
  // host-side state of the event stream
  int next_event = 0;
  std::vector<int> layer_event;       // event of the layer's current plan (-1 none)
  std::vector<int> layer_tokens;
  std::vector<int> fetch_event;       // event whose fetch was issued (-1 none)
  std::vector<int> forward_event;     // event whose FFN was enqueued (-1 none)
  // copy-engine thread: processes ring events 0, 1, 2, ... in order
  std::thread helper;
  std::atomic<bool> stop{false};
  std::atomic<long long> copied_events{0};  // events whose copies (and ready flag) are enqueued
  std::atomic<int> copy_status{0};          // first error of the copy thread (ft_status)
  std::atomic<bool> copies_paused{false};   // test knob: the copy thread serves no event while set
  std::mutex pool_mu;                       // guards pool and C against a resize while copies are issued
  // counters
  std::atomic<long long> launches{0}, memcpys{0};
  // timing
  std::atomic<bool> timing{false};   // read by the copy thread
  PhaseTimer timers[PHASE_COUNT];
  // step-graph capture: while set, ft_route_classify / ft_moe_forward record
  // external event nodes around their kernels into these arrays
  cudaStream_t capture_stream = nullptr;
  cudaEvent_t* cap_route_ev = nullptr;  // [2*L] begin/end per layer
  cudaEvent_t* cap_ffn_ev = nullptr;    // [2*L]
  cudaEvent_t* cap_fetch_ev = nullptr;  // [2*L] on the copy stream
};

namespace {

// Host banks that ft_cache_create registered, with the number of live caches
// using each.
std::mutex g_bank_mu;
std::map<const void*, int> g_bank_refs;

// Copy-engine thread.  Polls the stamp of ring entry e % kRing until it
// reads e (the route kernel writes every field first) and done_host until the
// FFN of event e - 2 has finished (its slots may be this event's victims),
// copies the event's misses from the host bank into their victim slots on the
// copy stream(s), then copies e into ready_flags[e % kRing] after them.  A
// ring entry is not overwritten before it is read: event e + kRing can only be
// routed after the FFN of event e + kRing - L - 1 or later ran (routing runs
// at most one step of L <= kRing - 2 layers ahead), which waited for this
// thread's flag of that event.
void helper_loop(ft_cache* c) {
  cudaSetDevice(c->device);
  long long e = 0;
  int idle = 0;
  while (!c->stop.load(std::memory_order_relaxed)) {
    if (c->copies_paused.load(std::memory_order_acquire)) {
      std::this_thread::sleep_for(std::chrono::microseconds(50));
      continue;
    }
    RingEntry* r = c->ring_host + (e % kRing);
    const int stamp = __atomic_load_n(&r->event, __ATOMIC_ACQUIRE);
    if (stamp > (int)e) {
      // Overrun: the entry was rewritten by a later event, which can only
      // happen after FFNs gave up waiting for this thread (their wait is
      // bounded).  Those events' copies are lost; report it and resume at the
      // oldest event still in the ring.
      int zero = 0;
      c->copy_status.compare_exchange_strong(zero, (int)FT_ERR_TIMEOUT);
      e = stamp - kRing + 1 > e ? stamp - kRing + 1 : e + 1;
      c->copied_events.store(e, std::memory_order_release);
      continue;
    }
    if (stamp != (int)e) {
      if (++idle > 20000) std::this_thread::sleep_for(std::chrono::microseconds(5));
      continue;
    }
    // the victims of event e may be slots that the FFN of event e - 2 reads
    if (e >= 2 && __atomic_load_n(&c->done_host[(e - 2) % kRing], __ATOMIC_ACQUIRE) != (int)(e - 2)) {
      if (++idle > 20000) std::this_thread::sleep_for(std::chrono::microseconds(5));
      continue;
    }
    idle = 0;
    int st = FT_OK;
    const int l = r->layer, n = r->n_miss;
    const bool tm = c->timing;
    std::lock_guard<std::mutex> pool_lock(c->pool_mu);
    if (tm) c->timers[PHASE_FETCH].begin(c->copy[0]);
    if (c->ncopy > 1) {  // the second stream starts with the first
      cudaEventRecord(c->copy_join, c->copy[0]);
      cudaStreamWaitEvent(c->copy[1], c->copy_join, 0);
    }
    for (int i = 0; i < n; ++i) {
      const int ex = r->miss_expert[i], sl = r->miss_slot[i];
      if (l < 0 || l >= c->L || ex < 0 || ex >= c->E || sl < 0 || sl >= c->C) {
        st = FT_ERR_CHECKED;
        break;
      }
      const int64_t blob = ((int64_t)l * c->E + ex) % c->cfg.bank_blobs;
      if (cudaMemcpyAsync(static_cast<uint8_t*>(c->pool) + (size_t)sl * c->eb, c->bank_host + (size_t)blob * c->eb,
                          c->eb, cudaMemcpyHostToDevice, c->copy[i % c->ncopy]) != cudaSuccess)
        st = FT_ERR_CUDA;
      ++c->memcpys;
    }
    if (c->ncopy > 1) {
      cudaEventRecord(c->copy_join, c->copy[1]);
      cudaStreamWaitEvent(c->copy[0], c->copy_join, 0);
    }
    c->flag_src[e % kRing] = (int)e;
    if (cudaMemcpyAsync(c->ready_flags + (e % kRing), c->flag_src + (e % kRing), sizeof(int32_t),
                        cudaMemcpyHostToDevice, c->copy[0]) != cudaSuccess)
      st = FT_ERR_CUDA;
    if (tm) c->timers[PHASE_FETCH].end(c->copy[0]);
    if (st != FT_OK) {
      int zero = 0;
      c->copy_status.compare_exchange_strong(zero, st);
    }
    c->copied_events.store(e + 1, std::memory_order_release);
    ++e;
  }
}

// Waits for a stream by polling: the copy thread may still have to enqueue
// the copies (and ready flags) that work on this stream waits for, so the
// waiting thread must not sit inside a blocking runtime call meanwhile.
cudaError_t wait_stream(cudaStream_t s) {
  for (;;) {
    const cudaError_t e = cudaStreamQuery(s);
    if (e != cudaErrorNotReady) return e;
    std::this_thread::sleep_for(std::chrono::microseconds(10));
  }
}

cudaError_t wait_event(cudaEvent_t ev) {
  for (;;) {
    const cudaError_t e = cudaEventQuery(ev);
    if (e != cudaErrorNotReady) return e;
    std::this_thread::sleep_for(std::chrono::microseconds(10));
  }
}

// SM pull on its own: a pull kernel on the copy stream after the layer's
// routing (and, when routing runs ahead, after the FFNs enqueued so far).
ft_status launch_pull(ft_cache* c, int layer) {
  CU(cudaStreamWaitEvent(c->copy[0], c->cls_ev[layer], 0));
  if (!c->route_follows_compute) {  // the victims' old contents may still be read by an enqueued FFN
    CU(cudaEventRecord(c->slots_free, c->compute));
    CU(cudaStreamWaitEvent(c->copy[0], c->slots_free, 0));
  }
  PullArgs p{};
  const Plan& pl = c->plans[layer];
  p.hdr = pl.hdr; p.miss_expert = pl.miss_expert; p.miss_slot = pl.miss_slot;
  p.layer = layer; p.E = c->E; p.bank_blobs = c->cfg.bank_blobs; p.bank = c->bank_dev;
  p.pool = c->pool; p.expert_bytes = (long long)c->eb;
  p.num_slots = (int)c->C; p.status = c->tab.status;
  const int ctas = c->cfg.pull_ctas > 0 ? c->cfg.pull_ctas : 64;
  if (c->timing) c->timers[PHASE_FETCH].begin(c->copy[0]);
  if (c->cap_fetch_ev) CU(cudaEventRecordWithFlags(c->cap_fetch_ev[2 * layer], c->copy[0], cudaEventRecordExternal));
  CU(launch_pull_misses(p, ctas, c->copy[0]));
  if (c->cap_fetch_ev) CU(cudaEventRecordWithFlags(c->cap_fetch_ev[2 * layer + 1], c->copy[0], cudaEventRecordExternal));
  if (c->timing) c->timers[PHASE_FETCH].end(c->copy[0]);
  ++c->launches;
  CU(cudaEventRecord(c->ready_ev[layer], c->copy[0]));
  return FT_OK;
}

ft_status flush_fetch(ft_cache* c) {
  if (c->pending_fetch < 0) return FT_OK;
  const int l = c->pending_fetch;
  c->pending_fetch = -1;
  return launch_pull(c, l);
}

ft_status sync_all(ft_cache* c) {
  if (c->pending_fetch >= 0) {  // a requested fetch is part of the work to finish
    const ft_status st = flush_fetch(c);
    if (st != FT_OK) return st;
  }
  CU(wait_stream(c->compute));  // FFNs (and graph replays) done
  CU(wait_stream(c->route));
  if (c->cfg.fetch_mode == FT_FETCH_COPY_ENGINE) {  // every routed event's copies must be enqueued
    CU(cudaMemcpyAsync(c->counter_host, c->tab.event_ctr, sizeof(int32_t), cudaMemcpyDeviceToHost, c->route));
    CU(wait_stream(c->route));
    const int routed = *c->counter_host;
    const auto t0 = std::chrono::steady_clock::now();
    while (c->copied_events.load(std::memory_order_acquire) < routed) {
      if (std::chrono::steady_clock::now() - t0 > std::chrono::seconds(10))
        return fail(FT_ERR_TIMEOUT, "copy thread did not reach event %d (at %lld) within 10 s", routed,
                    (long long)c->copied_events.load());
      std::this_thread::sleep_for(std::chrono::microseconds(10));
    }
  }
  for (int i = 0; i < c->ncopy; ++i) CU(wait_stream(c->copy[i]));
  CU(wait_stream(c->compute));
  const int cs = c->copy_status.load();
  if (cs != FT_OK) return fail((ft_status)cs, "a miss copy failed (%s)", ft_status_str((ft_status)cs));
  return FT_OK;
}

ft_status device_status(ft_cache* c) {
  int st = 0;
  CU(cudaMemcpy(&st, c->tab.status, sizeof st, cudaMemcpyDeviceToHost));
  if (st != 0) return fail((ft_status)st, "device status %d raised by an earlier call", st);
  return FT_OK;
}

ft_status alloc_tables(Tables& t, int64_t C, int num_keys, bool with_keys) {
  t.num_slots = (int32_t)C;
  t.num_keys = num_keys;
  if (with_keys) CU(cudaMalloc(&t.key_to_slot, sizeof(int32_t) * num_keys));
  CU(cudaMalloc(&t.slot_key, sizeof(int32_t) * C));
  CU(cudaMalloc(&t.slot_ts, sizeof(int32_t) * C));
  t.log_cap = log_capacity(C);
  CU(cudaMalloc(&t.log[0], sizeof(int2) * t.log_cap));
  CU(cudaMalloc(&t.log[1], sizeof(int2) * t.log_cap));
  CU(cudaMalloc(&t.pos, sizeof(int32_t) * C));
  CU(cudaMalloc(&t.log_cur, sizeof(int32_t) * 8));
  t.status = t.log_cur + 1;
  t.last_nu = t.log_cur + 2;
  t.event_ctr = t.log_cur + 3;
  t.pin_next = t.log_cur + 4;
  t.head = reinterpret_cast<uint32_t*>(t.log_cur + 5);
  t.tail = reinterpret_cast<uint32_t*>(t.log_cur + 6);
  CU(cudaMalloc(&t.stats, sizeof(long long) * ST_COUNT));
  return FT_OK;
}

void free_tables(Tables& t, bool with_keys) {
  if (with_keys) cudaFree(t.key_to_slot);
  cudaFree(t.slot_key);
  cudaFree(t.slot_ts);
  cudaFree(t.log[0]);
  cudaFree(t.log[1]);
  cudaFree(t.pos);
  cudaFree(t.log_cur);
  cudaFree(t.stats);
  Tables z{};
  z.key_to_slot = with_keys ? nullptr : t.key_to_slot;
  t = z;
}

// Device bytes of one cudaMalloc of n bytes, rounded to the allocation granularity.
uint64_t dev_alloc(uint64_t n) { return (n + 511) & ~uint64_t(511); }

// Checks the fields of a configuration that do not need a GPU; the message
// goes to ft_last_error.
ft_status check_config(const ft_cache_config& g) {
  if (g.num_layers < 1 || g.num_experts < 1 || g.num_experts > kMaxExperts)
    return fail(FT_ERR_INVALID_ARG, "num_layers must be >= 1 and num_experts in 1..%d", kMaxExperts);
  if (g.top_k < 1 || g.top_k > kMaxTopK || g.top_k > g.num_experts)
    return fail(FT_ERR_INVALID_ARG, "top_k must be in 1..min(num_experts, %d)", kMaxTopK);
  const size_t eb = blob_bytes(g.hidden, g.inter, g.wdtype);
  if (eb == 0) return fail(FT_ERR_INVALID_ARG, "unsupported hidden/inter/wdtype (%d, %d, %d)", g.hidden, g.inter, g.wdtype);
  if (eb % 16) return fail(FT_ERR_INVALID_ARG, "expert_bytes %zu is not a multiple of 16", eb);
  if (g.wdtype != FT_W_F32 && (g.hidden % 128 || g.inter % 128))
    return fail(FT_ERR_INVALID_ARG, "bf16/fp8 experts need hidden and inter multiples of 128");
  if (g.max_tokens < 1) return fail(FT_ERR_INVALID_ARG, "max_tokens must be >= 1");
  if ((long long)g.max_tokens * g.top_k > (1LL << 30)) return fail(FT_ERR_INVALID_ARG, "max_tokens * top_k too large");
  return FT_OK;
}

// Every device allocation ft_cache_create makes for C slots (the caller's pool
// aside), each rounded to the allocation granularity.
uint64_t cache_device_bytes(const ft_cache_config& g, int64_t C) {
  const uint64_t L = g.num_layers, E = g.num_experts, H = g.hidden, I = g.inter;
  const uint64_t rows = (uint64_t)g.max_tokens * g.top_k;
  uint64_t b = 0;
  // tables
  b += dev_alloc(4 * L * E) + 2 * dev_alloc(4 * (uint64_t)C) + 2 * dev_alloc(8 * (uint64_t)log_capacity(C)) +
       dev_alloc(4 * (uint64_t)C) + dev_alloc(32) + dev_alloc(8 * ST_COUNT);
  // plans
  const uint64_t per_plan = 4 * (PH_WORDS + 9 * E + 1 + 2 * rows) + 4 * rows;
  b += dev_alloc(((per_plan + 255) & ~uint64_t(255)) * L);
  // routing scratch, decode intermediate, FFN counters
  b += dev_alloc(4 * (kMaxExperts / 32) + 4 * kMaxExperts + 64);
  b += dev_alloc(4 * (uint64_t)std::min(g.max_tokens, kDecodeMaxTokens) * g.top_k * I);
  b += dev_alloc(16);
  if (g.max_tokens > kDecodeMaxTokens && prefill_supported((int)H, (int)I, g.wdtype, (int)E))
    b += dev_alloc(2 * rows * I) + dev_alloc(2 * rows * H) + dev_alloc(2 * rows * H) + dev_alloc(4 * rows) +
         dev_alloc(4 * E * (uint64_t)group_chunks((long long)rows));
  if (g.fetch_mode == FT_FETCH_COPY_ENGINE) b += dev_alloc(4 * kRing);
  return b;
}

int capacity_bound(const ft_cache* c) {
  const long long rows = (long long)c->max_tokens * c->k;
  return (int)(2 * std::min<long long>(rows, c->E));
}

// An NVTX range around a library call (shown by profilers that collect NVTX;
// free when none is attached), named after the call and carrying the layer.
struct NvtxRange {
  NvtxRange(const char* name, int layer) {
    nvtxEventAttributes_t ev = {};
    ev.version = NVTX_VERSION;
    ev.size = NVTX_EVENT_ATTRIB_STRUCT_SIZE;
    ev.messageType = NVTX_MESSAGE_TYPE_ASCII;
    ev.message.ascii = name;
    ev.payloadType = NVTX_PAYLOAD_TYPE_INT32;
    ev.payload.iValue = layer;
    nvtxRangePushEx(&ev);
  }
  ~NvtxRange() { nvtxRangePop(); }
};

}  // namespace

// ============================================================== the C ABI

extern "C" {

size_t ft_expert_bytes(int32_t hidden, int32_t inter, int32_t wdtype) { return blob_bytes(hidden, inter, wdtype); }

const char* ft_status_str(ft_status s) {
  switch (s) {
    case FT_OK: return "FT_OK";
    case FT_ERR_INVALID_ARG: return "FT_ERR_INVALID_ARG";
    case FT_ERR_CUDA: return "FT_ERR_CUDA";
    case FT_ERR_OOM: return "FT_ERR_OOM";
    case FT_ERR_CAPACITY: return "FT_ERR_CAPACITY";
    case FT_ERR_STATE: return "FT_ERR_STATE";
    case FT_ERR_TIMEOUT: return "FT_ERR_TIMEOUT";
    case FT_ERR_CHECKED: return "FT_ERR_CHECKED";
    case FT_ERR_UNSUPPORTED: return "FT_ERR_UNSUPPORTED";
  }
  return "FT_ERR_UNKNOWN";
}

const char* ft_last_error(void) { return g_last_error.c_str(); }

ft_status ft_cache_destroy(ft_cache* c) {
  if (!c) return FT_OK;
  cudaSetDevice(c->device);
  if (c->helper.joinable()) {
    c->stop = true;
    c->helper.join();
  }
  if (c->compute || c->copy[0]) {
    if (c->compute) wait_stream(c->compute);
    if (c->route) wait_stream(c->route);
    for (int i = 0; i < 2; ++i)
      if (c->copy[i]) cudaStreamSynchronize(c->copy[i]);
  }
  for (auto e : c->cls_ev) cudaEventDestroy(e);
  for (auto e : c->ready_ev) cudaEventDestroy(e);
  if (c->copy_join) cudaEventDestroy(c->copy_join);
  for (int i = 0; i < 2; ++i)
    if (c->copy[i]) cudaStreamDestroy(c->copy[i]);
  if (c->capture_stream) cudaStreamDestroy(c->capture_stream);
  if (c->route) cudaStreamDestroy(c->route);
  if (c->route_join) cudaEventDestroy(c->route_join);
  if (c->slots_free) cudaEventDestroy(c->slots_free);
  for (auto& ev : c->inflight)
    if (ev) cudaEventDestroy(ev);
  free_tables(c->tab, true);
  cudaFree(c->plan_mem);
  cudaFree(c->scr_mem);
  cudaFree(c->h_buf);
  cudaFree(c->pf_h);
  cudaFree(c->pf_xp);
  cudaFree(c->pf_yp);
  cudaFree(c->pf_pos);
  cudaFree(c->pf_hist);
  cudaFree(c->gbar);
  if (c->ring_host) cudaFreeHost(c->ring_host);
  if (c->flag_src) cudaFreeHost(c->flag_src);
  if (c->done_host) cudaFreeHost(c->done_host);
  if (c->counter_host) cudaFreeHost(c->counter_host);
  cudaFree(c->ready_flags);
  if (c->registered_bank) {
    std::lock_guard<std::mutex> lk(g_bank_mu);
    auto it = g_bank_refs.find(c->bank_host);
    if (it != g_bank_refs.end() && --it->second == 0) {
      cudaHostUnregister(const_cast<uint8_t*>(c->bank_host));
      g_bank_refs.erase(it);
    }
  }
  delete c;
  return FT_OK;
}

uint64_t ft_cache_overhead_bytes(const ft_cache_config* cfg, int64_t num_slots) {
  if (!cfg || num_slots < 1 || check_config(*cfg) != FT_OK) return 0;
  return cache_device_bytes(*cfg, num_slots);
}

ft_status ft_slots_for_budget(const ft_cache_config* cfg, uint64_t budget_bytes, int64_t* num_slots) {
  if (!cfg || !num_slots) return fail(FT_ERR_INVALID_ARG, "null config or output pointer");
  *num_slots = 0;
  const ft_status st = check_config(*cfg);
  if (st != FT_OK) return st;
  const uint64_t eb = blob_bytes(cfg->hidden, cfg->inter, cfg->wdtype);
  auto total = [&](int64_t C) { return (uint64_t)C * eb + cache_device_bytes(*cfg, C); };
  int64_t lo = 0, hi = (int64_t)std::min<uint64_t>(budget_bytes / eb, INT32_MAX / 2);
  while (lo < hi) {  // the most slots whose pool and tables fit the budget (total grows with C)
    const int64_t mid = lo + (hi - lo + 1) / 2;
    if (total(mid) <= budget_bytes) lo = mid;
    else hi = mid - 1;
  }
  const long long bound = 2 * std::min<long long>((long long)cfg->max_tokens * cfg->top_k, cfg->num_experts);
  if (lo < bound)
    return fail(FT_ERR_CAPACITY, "a budget of %llu bytes holds %lld slots, below the capacity bound %lld",
                (unsigned long long)budget_bytes, (long long)lo, bound);
  *num_slots = lo;
  return FT_OK;
}

ft_status ft_cache_create(const ft_cache_config* cfg, void* slot_pool, int64_t num_slots, void* compute_stream,
                          ft_cache** out) {
  if (!cfg || !out) return fail(FT_ERR_INVALID_ARG, "null config or output pointer");
  *out = nullptr;
  const ft_cache_config& g = *cfg;
  if (g.num_layers < 1 || g.num_experts < 1 || g.num_experts > kMaxExperts)
    return fail(FT_ERR_INVALID_ARG, "num_layers must be >= 1 and num_experts in 1..%d", kMaxExperts);
  if (g.top_k < 1 || g.top_k > kMaxTopK || g.top_k > g.num_experts)
    return fail(FT_ERR_INVALID_ARG, "top_k must be in 1..min(num_experts, %d)", kMaxTopK);
  const size_t eb = blob_bytes(g.hidden, g.inter, g.wdtype);
  if (eb == 0) return fail(FT_ERR_INVALID_ARG, "unsupported hidden/inter/wdtype (%d, %d, %d)", g.hidden, g.inter, g.wdtype);
  if (eb % 16) return fail(FT_ERR_INVALID_ARG, "expert_bytes %zu is not a multiple of 16", eb);
  if (g.wdtype != FT_W_F32 && (g.hidden % 128 || g.inter % 128))
    return fail(FT_ERR_INVALID_ARG, "bf16/fp8 experts need hidden and inter multiples of 128");
  if (g.max_tokens < 1) return fail(FT_ERR_INVALID_ARG, "max_tokens must be >= 1");
  if ((long long)g.max_tokens * g.top_k > (1LL << 30)) return fail(FT_ERR_INVALID_ARG, "max_tokens * top_k too large");
  if (g.fetch_mode != FT_FETCH_COPY_ENGINE && g.fetch_mode != FT_FETCH_SM_PULL)
    return fail(FT_ERR_INVALID_ARG, "unknown fetch_mode %d", g.fetch_mode);
  if (g.copy_streams < 0 || g.copy_streams > 2) return fail(FT_ERR_INVALID_ARG, "copy_streams must be 0, 1 or 2");
  if (g.fetch_warps < 0 || g.fetch_warps > kMaxFetchWarps)
    return fail(FT_ERR_INVALID_ARG, "fetch_warps must be 0..%d", kMaxFetchWarps);
  if (!g.host_bank || g.bank_blobs < 1 || g.bank_blobs > (int64_t)g.num_layers * g.num_experts)
    return fail(FT_ERR_INVALID_ARG, "host_bank null or bank_blobs outside 1..L*E");
  if (g.host_bank_bytes < (uint64_t)g.bank_blobs * eb)
    return fail(FT_ERR_INVALID_ARG, "host_bank_bytes %llu < bank_blobs * expert_bytes", (unsigned long long)g.host_bank_bytes);
  if (!slot_pool || (reinterpret_cast<uintptr_t>(slot_pool) & 255))
    return fail(FT_ERR_INVALID_ARG, "slot_pool must be a non-null 256-byte aligned device pointer");
  if (num_slots < 1 || num_slots > INT32_MAX / 2) return fail(FT_ERR_INVALID_ARG, "num_slots out of range");

  ft_cache* c = new ft_cache();
  c->cfg = g;
  c->L = g.num_layers; c->E = g.num_experts; c->k = g.top_k; c->H = g.hidden; c->I = g.inter;
  c->wdtype = g.wdtype; c->max_tokens = g.max_tokens; c->eb = eb;
  c->pool = slot_pool; c->C = num_slots;
  c->compute = static_cast<cudaStream_t>(compute_stream);
  c->ncopy = g.copy_streams == 2 ? 2 : 1;
  if (num_slots < capacity_bound(c)) {
    delete c;
    return fail(FT_ERR_CAPACITY, "num_slots %lld < 2 * min(max_tokens * top_k, num_experts) = %d", (long long)num_slots,
                2 * std::min<long long>((long long)g.max_tokens * g.top_k, g.num_experts));
  }
  ft_status st = [&]() -> ft_status {
    CU(cudaGetDevice(&c->device));
    cudaPointerAttributes pa{};
    CU(cudaPointerGetAttributes(&pa, slot_pool));
    if (pa.type != cudaMemoryTypeDevice) return fail(FT_ERR_INVALID_ARG, "slot_pool is not device memory");
    // host bank: pinned (registered) and mapped
    c->bank_host = static_cast<const uint8_t*>(g.host_bank);
    cudaPointerAttributes ha{};
    CU(cudaPointerGetAttributes(&ha, g.host_bank));
    if (ha.type == cudaMemoryTypeDevice || ha.type == cudaMemoryTypeManaged)
      return fail(FT_ERR_INVALID_ARG, "host_bank must be host memory");
    {
      // A bank the library registered stays registered while any cache uses it.
      std::lock_guard<std::mutex> lk(g_bank_mu);
      auto it = g_bank_refs.find(g.host_bank);
      if (it != g_bank_refs.end()) {
        ++it->second;
        c->registered_bank = true;
      } else if (ha.type != cudaMemoryTypeHost) {
        CU(cudaHostRegister(const_cast<void*>(g.host_bank), g.host_bank_bytes, cudaHostRegisterMapped));
        g_bank_refs[g.host_bank] = 1;
        c->registered_bank = true;
      }
    }
    void* dptr = nullptr;
    CU(cudaHostGetDevicePointer(&dptr, const_cast<void*>(g.host_bank), 0));
    c->bank_dev = dptr;
    // tables
    if (alloc_tables(c->tab, num_slots, c->L * c->E, true) != FT_OK) return FT_ERR_OOM;
    // plans
    const long long rows = (long long)g.max_tokens * g.top_k;
    const size_t per_plan = sizeof(int32_t) * (PH_WORDS + 9 * (size_t)c->E + 1 + 2 * rows) + sizeof(float) * rows;
    const size_t per_plan_al = (per_plan + 255) & ~size_t(255);
    CU(cudaMalloc(&c->plan_mem, per_plan_al * c->L));
    CU(cudaMemset(c->plan_mem, 0, per_plan_al * c->L));
    c->plans.resize(c->L);
    for (int l = 0; l < c->L; ++l) {
      int32_t* p = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(c->plan_mem) + per_plan_al * l);
      Plan& pl = c->plans[l];
      pl.hdr = p; p += PH_WORDS;
      pl.unique_expert = p; p += c->E;
      pl.unique_slot = p; p += c->E;
      pl.hit = p; p += c->E;
      pl.miss_expert = p; p += c->E;
      pl.miss_slot = p; p += c->E;
      pl.evicted_key = p; p += c->E;
      pl.e2u = p; p += c->E;
      pl.u_count = p; p += c->E;
      pl.u_offset = p; p += c->E + 1;
      pl.rows_by_u = p; p += rows;
      pl.topk_idx = p; p += rows;
      pl.topk_w = reinterpret_cast<float*>(p);
    }
    // routing scratch (zero; the kernel leaves it zero)
    const size_t scr_bytes = sizeof(uint32_t) * (kMaxExperts / 32) + sizeof(int32_t) * kMaxExperts + 64;
    CU(cudaMalloc(&c->scr_mem, scr_bytes));
    CU(cudaMemset(c->scr_mem, 0, scr_bytes));
    c->scr.bits = static_cast<uint32_t*>(c->scr_mem);
    c->scr.counts = reinterpret_cast<int32_t*>(c->scr.bits + kMaxExperts / 32);
    c->scr.ticket = reinterpret_cast<uint32_t*>(c->scr.counts + kMaxExperts);
    // decode intermediate
    const long long drows = (long long)std::min(g.max_tokens, kDecodeMaxTokens) * g.top_k;
    CU(cudaMalloc(&c->h_buf, sizeof(float) * drows * c->I));
    if (g.max_tokens > kDecodeMaxTokens && prefill_supported(c->H, c->I, c->wdtype, c->E)) {
      const long long prows = (long long)g.max_tokens * g.top_k;
      CU(cudaMalloc(&c->pf_h, sizeof(uint16_t) * prows * c->I));
      CU(cudaMalloc(&c->pf_xp, sizeof(uint16_t) * prows * c->H));
      CU(cudaMalloc(&c->pf_yp, sizeof(uint16_t) * prows * c->H));
      CU(cudaMalloc(&c->pf_pos, sizeof(int32_t) * prows));
      CU(cudaMalloc(&c->pf_hist, sizeof(int32_t) * c->E * group_chunks(prows)));
      prefill_init();
    }
    CU(cudaMalloc(&c->gbar, 4 * sizeof(unsigned)));
    CU(cudaMemset(c->gbar, 0, 3 * sizeof(unsigned)));
    CU(cudaMemset(c->gbar + 3, 0xff, sizeof(unsigned)));
    if (g.fetch_mode == FT_FETCH_COPY_ENGINE) {  // event ring (mapped host) and ready flags (device)
      CU(cudaHostAlloc(reinterpret_cast<void**>(&c->ring_host), sizeof(RingEntry) * kRing, cudaHostAllocMapped));
      memset(c->ring_host, 0, sizeof(RingEntry) * kRing);
      for (int i = 0; i < kRing; ++i) c->ring_host[i].event = -1;
      CU(cudaHostGetDevicePointer(reinterpret_cast<void**>(&c->ring_dev), c->ring_host, 0));
      CU(cudaHostAlloc(reinterpret_cast<void**>(&c->flag_src), sizeof(int32_t) * kRing, cudaHostAllocDefault));
      CU(cudaHostAlloc(reinterpret_cast<void**>(&c->done_host), sizeof(int32_t) * kRing, cudaHostAllocMapped));
      for (int i = 0; i < kRing; ++i) c->done_host[i] = -1;
      CU(cudaHostGetDevicePointer(reinterpret_cast<void**>(&c->done_dev), c->done_host, 0));
      CU(cudaHostAlloc(reinterpret_cast<void**>(&c->counter_host), sizeof(int32_t), cudaHostAllocDefault));
      CU(cudaMalloc(&c->ready_flags, sizeof(int32_t) * kRing));
      CU(cudaMemset(c->ready_flags, 0xff, sizeof(int32_t) * kRing));  // -1: no event yet
    }
    // streams and events
    for (int i = 0; i < c->ncopy; ++i) CU(cudaStreamCreateWithFlags(&c->copy[i], cudaStreamNonBlocking));
    CU(cudaStreamCreateWithFlags(&c->route, cudaStreamNonBlocking));
    CU(prefer_max_shared_route());
    CU(prefer_max_shared_fetch());
    CU(cudaEventCreateWithFlags(&c->route_join, cudaEventDisableTiming));
    CU(cudaEventCreateWithFlags(&c->slots_free, cudaEventDisableTiming));
    for (auto& ev : c->inflight) CU(cudaEventCreateWithFlags(&ev, cudaEventDisableTiming));
    CU(cudaEventCreateWithFlags(&c->copy_join, cudaEventDisableTiming));
    c->cls_ev.assign(c->L, nullptr);
    c->ready_ev.assign(c->L, nullptr);
    for (int l = 0; l < c->L; ++l) {
      CU(cudaEventCreateWithFlags(&c->cls_ev[l], cudaEventDisableTiming));
      CU(cudaEventCreateWithFlags(&c->ready_ev[l], cudaEventDisableTiming));
    }
    c->layer_event.assign(c->L, -1);
    c->layer_tokens.assign(c->L, 0);
    c->fetch_event.assign(c->L, -1);
    c->forward_event.assign(c->L, -1);
    CU(launch_init_tables(c->tab, c->L * c->E, c->compute));
    ++c->launches;
    CU(cudaStreamSynchronize(c->compute));
    if (g.fetch_mode == FT_FETCH_COPY_ENGINE) c->helper = std::thread(helper_loop, c);
    return FT_OK;
  }();
  if (st != FT_OK) {
    std::string msg = g_last_error;
    ft_cache_destroy(c);
    g_last_error = msg;
    return st;
  }
  *out = c;
  return FT_OK;
}

ft_status ft_route_classify(ft_cache* c, int32_t layer, const float* logits, int32_t T, int32_t* topk_idx,
                            float* topk_w) {
  NvtxRange nv("ft_route_classify", layer);
  if (!c) return fail(FT_ERR_INVALID_ARG, "null cache");
  if (layer < 0 || layer >= c->L) return fail(FT_ERR_INVALID_ARG, "layer %d out of range", layer);
  if (T < 0 || T > c->max_tokens) return fail(FT_ERR_INVALID_ARG, "T=%d outside 0..max_tokens=%d", T, c->max_tokens);
  if (T > 0 && !logits) return fail(FT_ERR_INVALID_ARG, "null logits");
  if (T > kDecodeMaxTokens && c->cfg.fetch_mode == FT_FETCH_COPY_ENGINE)  // its kernels do not wait for the copy thread
    return fail(FT_ERR_UNSUPPORTED, "T=%d > %d (prefill) needs the SM-pull fetch mode", T, kDecodeMaxTokens);
  const int t = c->next_event;
  // a fetched plan must be consumed by its FFN before the layer is re-planned
  if (c->fetch_event[layer] >= 0 && c->fetch_event[layer] == c->layer_event[layer] &&
      c->forward_event[layer] != c->layer_event[layer])
    return fail(FT_ERR_STATE, "layer %d: fetched plan not yet forwarded", layer);
  // pipelining depth: every fetched event older than t-1 must have its FFN enqueued
  for (int l = 0; l < c->L; ++l)
    if (c->fetch_event[l] >= 0 && c->fetch_event[l] <= t - 2 && c->forward_event[l] != c->fetch_event[l])
      return fail(FT_ERR_STATE, "layer %d (event %d) fetched but not forwarded; only one layer may run ahead", l,
                  c->fetch_event[l]);
  RouteArgs a{};
  a.logits = logits; a.T = T; a.E = c->E; a.k = c->k; a.layer = layer;
  a.out_idx = topk_idx; a.out_w = topk_w;
  a.tab = c->tab; a.plan = c->plans[layer]; a.scr = c->scr;
  a.ring = c->ring_dev;
  a.expert_bytes = (long long)c->eb;
  a.build_rows = (long long)T * c->k <= kMaxExperts;
  // The route stream starts after everything the caller has enqueued on the
  // compute stream so far: the logits, and in the double-buffered schedule the
  // FFN of event t-2 (whose slots this event may evict).
  if (c->route_follows_compute) {
    CU(cudaEventRecord(c->route_join, c->compute));
    CU(cudaStreamWaitEvent(c->route, c->route_join, 0));
  }
  if (c->timing) c->timers[PHASE_ROUTE].begin(c->route);
  if (c->cap_route_ev) CU(cudaEventRecordWithFlags(c->cap_route_ev[2 * layer], c->route, cudaEventRecordExternal));
  CU(launch_route_classify(a, c->route));
  if (c->cap_route_ev) CU(cudaEventRecordWithFlags(c->cap_route_ev[2 * layer + 1], c->route, cudaEventRecordExternal));
  if (c->timing) c->timers[PHASE_ROUTE].end(c->route);
  ++c->launches;
  CU(cudaEventRecord(c->cls_ev[layer], c->route));
  c->layer_event[layer] = t;
  c->layer_tokens[layer] = T;
  c->next_event = t + 1;
  return FT_OK;
}


ft_status ft_fetch_misses(ft_cache* c, int32_t layer) {
  NvtxRange nv("ft_fetch_misses", layer);
  if (!c) return fail(FT_ERR_INVALID_ARG, "null cache");
  if (layer < 0 || layer >= c->L) return fail(FT_ERR_INVALID_ARG, "layer %d out of range", layer);
  const int ev = c->layer_event[layer];
  if (ev < 0 || c->fetch_event[layer] == ev) return fail(FT_ERR_STATE, "layer %d has no classification awaiting fetch", layer);
  if (c->cfg.fetch_mode == FT_FETCH_COPY_ENGINE) {
    // nothing to enqueue: the copy thread picks the event up from the ring
  } else {
    // deferred: the next forward of another layer copies these misses inside
    // its kernel; at most one fetch waits
    ft_status st = flush_fetch(c);
    if (st != FT_OK) return st;
    c->pending_fetch = layer;
  }
  c->fetch_event[layer] = ev;
  return FT_OK;
}

ft_status ft_moe_forward(ft_cache* c, int32_t layer, const void* x, int32_t T, void* y) {
  NvtxRange nv("ft_moe_forward", layer);
  if (!c) return fail(FT_ERR_INVALID_ARG, "null cache");
  if (layer < 0 || layer >= c->L) return fail(FT_ERR_INVALID_ARG, "layer %d out of range", layer);
  const int ev = c->layer_event[layer];
  if (ev < 0 || c->fetch_event[layer] != ev || c->forward_event[layer] == ev)
    return fail(FT_ERR_STATE, "layer %d: forward needs a classified and fetched plan", layer);
  if (T != c->layer_tokens[layer]) return fail(FT_ERR_INVALID_ARG, "T=%d differs from the plan's T=%d", T, c->layer_tokens[layer]);
  if (T > 0 && (!x || !y)) return fail(FT_ERR_INVALID_ARG, "null x or y");
  if (c->cfg.fetch_mode == FT_FETCH_COPY_ENGINE) {
    // the FFN reads the plan written by route_classify; its slots are waited
    // for inside the kernel (ready flag set after the copies)
    CU(cudaStreamWaitEvent(c->compute, c->cls_ev[layer], 0));
  } else {
    if (c->pending_fetch == layer || T == 0 || T > kDecodeMaxTokens || !c->fused_ok) {
      ft_status st = flush_fetch(c);  // this layer's own fetch, or no fused kernel to carry it
      if (st != FT_OK) return st;
    }
    CU(cudaStreamWaitEvent(c->compute, c->ready_ev[layer], 0));
  }
  c->forward_event[layer] = ev;
  if (T == 0) {
    if (c->cfg.fetch_mode == FT_FETCH_COPY_ENGINE) {  // no FFN kernel: the copy thread still needs the signal
      FfnArgs f0{};
      f0.hdr = c->plans[layer].hdr;
      f0.done_host = c->done_dev;
      CU(launch_signal_done(f0, c->compute));
      ++c->launches;
    }
    return FT_OK;
  }
  const Plan& pl = c->plans[layer];
  if (T > kDecodeMaxTokens) {  // prefill: grouped GEMMs
    if (!c->pf_yp)
      return fail(FT_ERR_UNSUPPORTED, "T=%d > %d: the prefill path needs bf16 or fp8 weights (H %% 128, I %% 128)", T,
                  kDecodeMaxTokens);
    PrefillArgs p{};
    p.hdr = pl.hdr; p.unique_expert = pl.unique_expert; p.unique_slot = pl.unique_slot; p.u_offset = pl.u_offset;
    p.topk_idx = pl.topk_idx; p.topk_w = pl.topk_w; p.rows_by_u = pl.rows_by_u; p.pos = c->pf_pos;
    p.hist = c->pf_hist;
    p.x = x; p.xp = c->pf_xp; p.h = c->pf_h; p.yp = c->pf_yp; p.y = static_cast<float*>(y);
    p.pool = static_cast<const uint8_t*>(c->pool); p.expert_bytes = (long long)c->eb;
    p.H = c->H; p.I = c->I; p.k = c->k; p.T = T; p.E = c->E; p.status = c->tab.status; p.wdtype = c->wdtype;
    const bool tm = c->timing;
    if (tm) c->timers[PHASE_FFN].begin(c->compute);
    if (c->cap_ffn_ev) CU(cudaEventRecordWithFlags(c->cap_ffn_ev[2 * layer], c->compute, cudaEventRecordExternal));
    int n = 0;
    cudaEvent_t marks[4] = {};
    const bool gm = tm && c->timers[PHASE_GEMM1].reserve(&marks[0], &marks[1]) &&
                    c->timers[PHASE_GEMM2].reserve(&marks[2], &marks[3]);
    const cudaError_t e = launch_prefill_ffn(p, (int)c->C, c->compute, &n, gm ? marks : nullptr);
    if (e != cudaSuccess) return fail(FT_ERR_CUDA, "prefill FFN launch: %s", cudaGetErrorString(e));
    c->launches += n;
    if (c->cap_ffn_ev) CU(cudaEventRecordWithFlags(c->cap_ffn_ev[2 * layer + 1], c->compute, cudaEventRecordExternal));
    if (tm) c->timers[PHASE_FFN].end(c->compute);
    return FT_OK;
  }
  FfnArgs f{};
  f.hdr = pl.hdr; f.unique_slot = pl.unique_slot; f.hit = pl.hit; f.u_offset = pl.u_offset; f.rows_by_u = pl.rows_by_u;
  f.topk_w = pl.topk_w; f.x = x; f.y = static_cast<float*>(y); f.pool = static_cast<const uint8_t*>(c->pool);
  f.expert_bytes = (long long)c->eb; f.num_slots = (int)c->C;
  f.H = c->H; f.I = c->I; f.k = c->k; f.T = T; f.wdtype = c->wdtype; f.h = c->h_buf;
  f.max_unique = std::min(T * c->k, c->E);
  f.status = c->tab.status;
  f.gbar = c->gbar;
  f.ready_flags = c->cfg.fetch_mode == FT_FETCH_COPY_ENGINE ? c->ready_flags : nullptr;
  f.done_host = c->cfg.fetch_mode == FT_FETCH_COPY_ENGINE ? c->done_dev : nullptr;
  // the two kernels are timed as one unit: an event between them would cut
  // the programmatic dependency that lets the down kernel start early
  const bool tm = c->timing;
  const int nx = c->pending_fetch;  // fetched inside this FFN's kernel, if it launches
  if (nx >= 0) {
    CU(cudaStreamWaitEvent(c->compute, c->cls_ev[nx], 0));  // its miss list
    const Plan& pn = c->plans[nx];
    f.nx.hdr = pn.hdr; f.nx.miss_expert = pn.miss_expert; f.nx.miss_slot = pn.miss_slot;
    f.nx.layer = nx; f.nx.E = c->E; f.nx.bank_blobs = c->cfg.bank_blobs; f.nx.bank = c->bank_dev;
    f.nx.pool = c->pool; f.nx.expert_bytes = (long long)c->eb;
    f.nx.num_slots = (int)c->C; f.nx.status = c->tab.status;
    f.fetch_warps = c->cfg.fetch_warps > 0 ? c->cfg.fetch_warps : kDefaultFetchWarps;
    if (c->cap_fetch_ev) CU(cudaEventRecordWithFlags(c->cap_fetch_ev[2 * nx], c->compute, cudaEventRecordExternal));
  }
  if (tm) c->timers[PHASE_FFN].begin(c->compute);
  if (c->cap_ffn_ev) CU(cudaEventRecordWithFlags(c->cap_ffn_ev[2 * layer], c->compute, cudaEventRecordExternal));
  cudaError_t e = c->fused_ok ? launch_decode_ffn_fused(f, c->compute) : cudaErrorNotSupported;
  if (e == cudaSuccess) {
    ++c->launches;
    if (nx >= 0) {
      c->pending_fetch = -1;
      if (c->cap_fetch_ev)
        CU(cudaEventRecordWithFlags(c->cap_fetch_ev[2 * nx + 1], c->compute, cudaEventRecordExternal));
      CU(cudaEventRecord(c->ready_ev[nx], c->compute));
    }
  } else {
    if (e != cudaErrorNotSupported) {
      cudaGetLastError();  // clear a launch-configuration error, then take the two-kernel path from now on
      c->fused_ok = false;
    }
    e = launch_decode_gateup(f, c->compute);
    if (e != cudaSuccess) return fail(FT_ERR_CUDA, "gate/up launch: %s", cudaGetErrorString(e));
    ++c->launches;
    e = launch_decode_down(f, c->compute);
    if (e != cudaSuccess) return fail(FT_ERR_CUDA, "down launch: %s", cudaGetErrorString(e));
    ++c->launches;
    if (f.done_host) {
      e = launch_signal_done(f, c->compute);
      if (e != cudaSuccess) return fail(FT_ERR_CUDA, "done-signal launch: %s", cudaGetErrorString(e));
      ++c->launches;
    }
  }
  if (c->cap_ffn_ev) CU(cudaEventRecordWithFlags(c->cap_ffn_ev[2 * layer + 1], c->compute, cudaEventRecordExternal));
  if (tm) c->timers[PHASE_FFN].end(c->compute);
  if (nx >= 0 && c->pending_fetch == nx) return flush_fetch(c);  // the two-kernel path did not carry it
  return FT_OK;
}

ft_status ft_cache_resize(ft_cache* c, void* new_pool, int64_t new_num_slots) {
  NvtxRange nv("ft_cache_resize", (int)new_num_slots);
  if (!c) return fail(FT_ERR_INVALID_ARG, "null cache");
  if (!new_pool || (reinterpret_cast<uintptr_t>(new_pool) & 255))
    return fail(FT_ERR_INVALID_ARG, "new_pool must be a non-null 256-byte aligned device pointer");
  if (new_num_slots < 1 || new_num_slots > INT32_MAX / 2) return fail(FT_ERR_INVALID_ARG, "new_num_slots out of range");
  if (new_num_slots < capacity_bound(c))
    return fail(FT_ERR_CAPACITY, "new_num_slots %lld below the capacity bound %d", (long long)new_num_slots, capacity_bound(c));
  for (int l = 0; l < c->L; ++l)
    if (c->fetch_event[l] >= 0 && c->fetch_event[l] == c->layer_event[l] && c->forward_event[l] != c->fetch_event[l])
      return fail(FT_ERR_STATE, "layer %d has a fetched plan whose FFN was not enqueued", l);
  ft_status s = sync_all(c);  // the safe point
  if (s != FT_OK) return s;
  cudaPointerAttributes pa{};
  CU(cudaPointerGetAttributes(&pa, new_pool));
  if (pa.type != cudaMemoryTypeDevice) return fail(FT_ERR_INVALID_ARG, "new_pool is not device memory");
  Tables nt{};
  nt.key_to_slot = c->tab.key_to_slot;
  if (alloc_tables(nt, new_num_slots, c->L * c->E, false) != FT_OK) {
    free_tables(nt, false);
    return FT_ERR_OOM;
  }
  int32_t* moves = nullptr;
  const int64_t max_moves = std::max<int64_t>(new_num_slots, 1);
  cudaError_t e = cudaMalloc(&moves, sizeof(int32_t) * (2 * max_moves + 1));
  if (e != cudaSuccess) {
    free_tables(nt, false);
    return fail(FT_ERR_OOM, "resize move list: %s", cudaGetErrorString(e));
  }
  ResizeArgs ra{};
  ra.old_tab = c->tab; ra.new_tab = nt; ra.num_keys = c->L * c->E; ra.E = c->E;
  ra.moves = moves + 1; ra.n_moves = moves; ra.copy_all = new_pool != c->pool;
  int n = 0;
  e = launch_resize_tables(ra, c->compute, &n);
  c->launches += n;
  if (e == cudaSuccess) {
    e = launch_move_blobs(ra.moves, ra.n_moves, (int)max_moves, c->pool, new_pool, (long long)c->eb, c->compute);
    ++c->launches;
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(c->compute);
  cudaFree(moves);
  if (e != cudaSuccess) {
    free_tables(nt, false);
    return fail(FT_ERR_CUDA, "resize: %s", cudaGetErrorString(e));
  }
  free_tables(c->tab, false);
  c->tab = nt;
  {
    std::lock_guard<std::mutex> lk(c->pool_mu);
    c->pool = new_pool;
    c->C = new_num_slots;
  }
  for (int l = 0; l < c->L; ++l) {
    c->layer_event[l] = -1;
    c->fetch_event[l] = -1;
    c->forward_event[l] = -1;
  }
  return FT_OK;
}

ft_status ft_synchronize(ft_cache* c) {
  if (!c) return fail(FT_ERR_INVALID_ARG, "null cache");
  ft_status s = sync_all(c);
  if (s != FT_OK) return s;
  return device_status(c);
}

ft_status ft_get_plan(ft_cache* c, int32_t layer, ft_plan_info* info, int32_t* unique_expert, int32_t* unique_slot,
                      uint8_t* hit, int32_t* miss_expert, int32_t* miss_slot, int32_t* evicted_key) {
  if (!c) return fail(FT_ERR_INVALID_ARG, "null cache");
  if (layer < 0 || layer >= c->L) return fail(FT_ERR_INVALID_ARG, "layer %d out of range", layer);
  ft_status s = sync_all(c);
  if (s != FT_OK) return s;
  const Plan& pl = c->plans[layer];
  int32_t hdr[PH_WORDS];
  CU(cudaMemcpy(hdr, pl.hdr, sizeof hdr, cudaMemcpyDeviceToHost));
  if (info) {
    info->event = hdr[PH_EVENT];
    info->n_tokens = hdr[PH_TOKENS];
    info->n_unique = hdr[PH_UNIQUE];
    info->n_miss = hdr[PH_MISS];
  }
  const int nu = hdr[PH_UNIQUE], nm = hdr[PH_MISS];
  if (unique_expert && nu) CU(cudaMemcpy(unique_expert, pl.unique_expert, sizeof(int32_t) * nu, cudaMemcpyDeviceToHost));
  if (unique_slot && nu) CU(cudaMemcpy(unique_slot, pl.unique_slot, sizeof(int32_t) * nu, cudaMemcpyDeviceToHost));
  if (hit && nu) {
    std::vector<int32_t> h(nu);
    CU(cudaMemcpy(h.data(), pl.hit, sizeof(int32_t) * nu, cudaMemcpyDeviceToHost));
    for (int i = 0; i < nu; ++i) hit[i] = (uint8_t)h[i];
  }
  if (miss_expert && nm) CU(cudaMemcpy(miss_expert, pl.miss_expert, sizeof(int32_t) * nm, cudaMemcpyDeviceToHost));
  if (miss_slot && nm) CU(cudaMemcpy(miss_slot, pl.miss_slot, sizeof(int32_t) * nm, cudaMemcpyDeviceToHost));
  if (evicted_key && nm) CU(cudaMemcpy(evicted_key, pl.evicted_key, sizeof(int32_t) * nm, cudaMemcpyDeviceToHost));
  return FT_OK;
}

ft_status ft_get_tables(ft_cache* c, int32_t* key_to_slot, int32_t* slot_key, int32_t* slot_ts) {
  if (!c) return fail(FT_ERR_INVALID_ARG, "null cache");
  ft_status s = sync_all(c);
  if (s != FT_OK) return s;
  if (key_to_slot) CU(cudaMemcpy(key_to_slot, c->tab.key_to_slot, sizeof(int32_t) * c->L * c->E, cudaMemcpyDeviceToHost));
  if (slot_key) CU(cudaMemcpy(slot_key, c->tab.slot_key, sizeof(int32_t) * c->C, cudaMemcpyDeviceToHost));
  if (slot_ts) CU(cudaMemcpy(slot_ts, c->tab.slot_ts, sizeof(int32_t) * c->C, cudaMemcpyDeviceToHost));
  return FT_OK;
}

ft_status ft_get_stats(ft_cache* c, ft_stats* out) {
  if (!c || !out) return fail(FT_ERR_INVALID_ARG, "null argument");
  ft_status s = sync_all(c);
  if (s != FT_OK) return s;
  long long st[ST_COUNT];
  CU(cudaMemcpy(st, c->tab.stats, sizeof st, cudaMemcpyDeviceToHost));
  out->events = st[ST_EVENTS];
  out->unique_experts = st[ST_UNIQUE];
  out->hits = st[ST_HITS];
  out->misses = st[ST_MISSES];
  out->evictions = st[ST_EVICT];
  out->bytes_fetched = st[ST_BYTES];
  out->kernel_launches = c->launches.load();
  out->memcpy_calls = c->memcpys.load();
  return device_status(c);
}

ft_status ft_reset_stats(ft_cache* c) {
  if (!c) return fail(FT_ERR_INVALID_ARG, "null cache");
  ft_status s = sync_all(c);
  if (s != FT_OK) return s;
  CU(cudaMemset(c->tab.stats, 0, sizeof(long long) * ST_COUNT));
  c->launches = 0;
  c->memcpys = 0;
  return FT_OK;
}

ft_status ft_get_pool(ft_cache* c, void** pool, int64_t* num_slots) {
  if (!c) return fail(FT_ERR_INVALID_ARG, "null cache");
  if (pool) *pool = c->pool;
  if (num_slots) *num_slots = c->C;
  return FT_OK;
}

ft_status ft_debug_pause_copies(ft_cache* c, int32_t paused) {
  if (!c) return fail(FT_ERR_INVALID_ARG, "null cache");
  if (c->cfg.fetch_mode != FT_FETCH_COPY_ENGINE) return fail(FT_ERR_STATE, "the cache has no copy thread");
  c->copies_paused.store(paused != 0, std::memory_order_release);
  return FT_OK;
}

int32_t ft_checked_build(void) { return kChecked ? 1 : 0; }

ft_status ft_host_bank_alloc(uint64_t bytes, void** host) {
  if (!host || bytes == 0) return fail(FT_ERR_INVALID_ARG, "null out pointer or zero bytes");
  *host = nullptr;
  const cudaError_t e = cudaHostAlloc(host, bytes, cudaHostAllocPortable | cudaHostAllocMapped);
  if (e != cudaSuccess) {
    cudaGetLastError();
    *host = nullptr;
    return fail(FT_ERR_OOM, "cudaHostAlloc of %llu bytes: %s", (unsigned long long)bytes, cudaGetErrorString(e));
  }
  return FT_OK;
}

ft_status ft_host_bank_free(void* host) {
  if (!host) return FT_OK;
  CU(cudaFreeHost(host));
  return FT_OK;
}

ft_status ft_debug_set_key_slot(ft_cache* c, int32_t key, int32_t slot) {
  if (!c) return fail(FT_ERR_INVALID_ARG, "null cache");
  if (!kChecked) return fail(FT_ERR_STATE, "only the bounds-checked build takes a corrupted slot table");
  if (key < 0 || (long long)key >= (long long)c->L * c->E) return fail(FT_ERR_INVALID_ARG, "key %d out of range", key);
  CU(cudaDeviceSynchronize());
  CU(cudaMemcpy(c->tab.key_to_slot + key, &slot, sizeof slot, cudaMemcpyHostToDevice));
  return FT_OK;
}

ft_status ft_get_copy_stream(ft_cache* c, void** stream) {
  if (!c || !stream) return fail(FT_ERR_INVALID_ARG, "null argument");
  *stream = c->copy[0];
  return FT_OK;
}

ft_status ft_timing_enable(ft_cache* c, int32_t on) {
  if (!c) return fail(FT_ERR_INVALID_ARG, "null cache");
  ft_status s = sync_all(c);
  if (s != FT_OK) return s;
  for (auto& t : c->timers) {
    t.reset();
    // the events exist before the first timed phase: creating a pool of them
    // inside a timed window would count that host time as GPU time
    if (on && !t.ensure()) return fail(FT_ERR_CUDA, "creating timing events failed");
  }
  c->timing = on != 0;
  return FT_OK;
}

ft_status ft_get_timing(ft_cache* c, ft_timing* out) {
  if (!c || !out) return fail(FT_ERR_INVALID_ARG, "null argument");
  ft_status s = sync_all(c);
  if (s != FT_OK) return s;
  for (auto& t : c->timers) t.collect();
  out->route_ms = c->timers[PHASE_ROUTE].total_ms; out->route_n = c->timers[PHASE_ROUTE].n;
  out->fetch_ms = c->timers[PHASE_FETCH].total_ms; out->fetch_n = c->timers[PHASE_FETCH].n;
  out->ffn_ms = c->timers[PHASE_FFN].total_ms; out->ffn_n = c->timers[PHASE_FFN].n;
  out->gemm1_ms = c->timers[PHASE_GEMM1].total_ms; out->gemm1_n = c->timers[PHASE_GEMM1].n;
  out->gemm2_ms = c->timers[PHASE_GEMM2].total_ms; out->gemm2_n = c->timers[PHASE_GEMM2].n;
  return FT_OK;
}

// ----------------------------------------------------------------- step graphs

struct ft_step_graph {
  ft_cache* c = nullptr;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  int L = 0;
  long long kernels = 0;  // kernels per launch
  std::vector<cudaEvent_t> ev;  // [0,2L) route, [2L,4L) ffn, [4L,6L) fetch begin/end; then step begin/end
  bool timing = false;
  bool fetch_events = false;  // false in copy-engine mode: the copy thread's copies are not graph nodes
  bool launched = false;
};

ft_status ft_step_graph_destroy(ft_step_graph* g) {
  if (!g) return FT_OK;
  if (g->c) cudaSetDevice(g->c->device);
  if (g->launched && g->c) wait_stream(g->c->compute);
  if (g->exec) cudaGraphExecDestroy(g->exec);
  if (g->graph) cudaGraphDestroy(g->graph);
  for (auto e : g->ev) cudaEventDestroy(e);
  delete g;
  return FT_OK;
}

ft_status ft_step_graph_create(ft_cache* c, const float* const* logits, const void* const* x, float* const* y,
                               int32_t T, int32_t double_buffer, int32_t timing, ft_step_graph** out) {
  if (!c || !out || !logits || !x || !y) return fail(FT_ERR_INVALID_ARG, "null argument");
  *out = nullptr;
  if (T < 0 || T > c->max_tokens) return fail(FT_ERR_INVALID_ARG, "T=%d outside 0..max_tokens", T);
  for (int l = 0; l < c->L; ++l) {
    if (T > 0 && (!logits[l] || !x[l] || !y[l])) return fail(FT_ERR_INVALID_ARG, "null buffer for layer %d", l);
    if (c->fetch_event[l] >= 0 && c->fetch_event[l] == c->layer_event[l] && c->forward_event[l] != c->fetch_event[l])
      return fail(FT_ERR_STATE, "layer %d has a fetched plan whose FFN was not enqueued", l);
  }
  ft_status st = sync_all(c);
  if (st != FT_OK) return st;
  ft_step_graph* g = new ft_step_graph();
  g->c = c;
  g->L = c->L;
  g->timing = timing != 0;
  const int nev = 6 * c->L + 2;
  g->ev.assign(nev, nullptr);
  for (auto& e : g->ev)
    if (cudaEventCreate(&e) != cudaSuccess) {
      ft_step_graph_destroy(g);
      return fail(FT_ERR_CUDA, "cudaEventCreate failed");
    }
  if (!c->capture_stream && cudaStreamCreateWithFlags(&c->capture_stream, cudaStreamNonBlocking) != cudaSuccess) {
    ft_step_graph_destroy(g);
    return fail(FT_ERR_CUDA, "capture stream creation failed");
  }
  cudaStream_t saved_compute = c->compute;
  const bool saved_timing = c->timing;
  const long long launches0 = c->launches.load();
  c->compute = c->capture_stream;
  c->timing = false;
  if (g->timing) {
    c->cap_route_ev = g->ev.data();
    c->cap_ffn_ev = g->ev.data() + 2 * c->L;
    c->cap_fetch_ev = g->ev.data() + 4 * c->L;
    g->fetch_events = c->cfg.fetch_mode == FT_FETCH_SM_PULL;
  }
  auto restore = [&]() {
    c->compute = saved_compute;
    c->timing = saved_timing;
    c->route_follows_compute = true;
    c->cap_route_ev = nullptr;
    c->cap_ffn_ev = nullptr;
    c->cap_fetch_ev = nullptr;
  };
  cudaError_t e = cudaStreamBeginCapture(c->capture_stream, cudaStreamCaptureModeRelaxed);
  if (e != cudaSuccess) {
    restore();
    ft_step_graph_destroy(g);
    return fail(FT_ERR_CUDA, "cudaStreamBeginCapture: %s", cudaGetErrorString(e));
  }
  if (g->timing) cudaEventRecordWithFlags(g->ev[6 * c->L], c->capture_stream, cudaEventRecordExternal);
  if (c->cfg.fetch_mode == FT_FETCH_SM_PULL || c->L + 2 <= kRing) {
    // Routing runs ahead on the route stream from the step's start (the
    // logits are inputs of the graph).  Each pull kernel waits for its routing
    // and for the FFN enqueued before it; in copy-engine mode the copy thread
    // waits for the FFN of event t - 2 before it copies event t's misses.
    e = cudaEventRecord(c->route_join, c->compute);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(c->route, c->route_join, 0);
    c->route_follows_compute = false;
  }
  auto route = [&](int l) -> ft_status {
    ft_status s1 = ft_route_classify(c, l, logits[l], T, nullptr, nullptr);
    return s1 != FT_OK ? s1 : ft_fetch_misses(c, l);
  };
  st = e == cudaSuccess ? FT_OK : fail(FT_ERR_CUDA, "route stream join: %s", cudaGetErrorString(e));
  if (st == FT_OK && double_buffer) {
    st = route(0);
    for (int l = 0; l < c->L && st == FT_OK; ++l) {
      if (l + 1 < c->L) st = route(l + 1);
      if (st == FT_OK) st = ft_moe_forward(c, l, x[l], T, y[l]);
    }
  } else if (st == FT_OK) {
    for (int l = 0; l < c->L && st == FT_OK; ++l) {
      st = route(l);
      if (st == FT_OK) st = ft_moe_forward(c, l, x[l], T, y[l]);
    }
  }
  if (st == FT_OK && c->pending_fetch >= 0) st = flush_fetch(c);  // inside the capture
  if (g->timing) cudaEventRecordWithFlags(g->ev[6 * c->L + 1], c->capture_stream, cudaEventRecordExternal);
  const std::string msg = g_last_error;
  e = cudaStreamEndCapture(c->capture_stream, &g->graph);
  restore();
  g->kernels = c->launches.load() - launches0;
  c->launches = launches0;
  if (st != FT_OK || e != cudaSuccess) {
    ft_step_graph_destroy(g);
    if (st != FT_OK) return fail(st, "capture: %s", msg.c_str());
    return fail(FT_ERR_CUDA, "cudaStreamEndCapture: %s", cudaGetErrorString(e));
  }
  e = cudaGraphInstantiate(&g->exec, g->graph, 0);
  if (e == cudaSuccess) e = cudaGraphUpload(g->exec, c->compute);
  if (e != cudaSuccess) {
    ft_step_graph_destroy(g);
    return fail(FT_ERR_CUDA, "cudaGraphInstantiate: %s", cudaGetErrorString(e));
  }
  *out = g;
  return FT_OK;
}

ft_status ft_step_graph_launch(ft_step_graph* g) {
  NvtxRange nv("ft_step_graph_launch", -1);
  if (!g || !g->exec) return fail(FT_ERR_INVALID_ARG, "null step graph");
  ft_cache* c = g->c;
  const bool ce = c->cfg.fetch_mode == FT_FETCH_COPY_ENGINE;
  cudaEvent_t done = c->inflight[c->graph_launches % 2];
  if (ce && c->graph_launches >= 2) CU(wait_event(done));
  CU(cudaGraphLaunch(g->exec, c->compute));
  if (ce) CU(cudaEventRecord(done, c->compute));
  ++c->graph_launches;
  g->c->launches += g->kernels;
  g->launched = true;
  return FT_OK;
}

ft_status ft_step_graph_trace(ft_step_graph* g, double* t_ms) {
  if (!g || !t_ms) return fail(FT_ERR_INVALID_ARG, "null argument");
  if (!g->timing || !g->launched) return fail(FT_ERR_STATE, "graph was created without timing or never launched");
  const int L = g->L;
  CU(wait_event(g->ev[6 * L + 1]));
  float ms = 0.0f;
  for (int l = 0; l < L; ++l)
    for (int j = 0; j < 6; ++j) {  // route begin/end, fetch begin/end, ffn begin/end
      static const int base[3] = {0, 4, 2};  // event arrays: route [0, 2L), ffn [2L, 4L), fetch [4L, 6L)
      const int idx = base[j / 2] * L + 2 * l + (j & 1);
      if (j / 2 == 1 && !g->fetch_events) {
        t_ms[6 * l + j] = -1.0;
        continue;
      }
      CU(cudaEventElapsedTime(&ms, g->ev[6 * L], g->ev[idx]));
      t_ms[6 * l + j] = ms;
    }
  return FT_OK;
}

ft_status ft_step_graph_timing(ft_step_graph* g, double* route_ms, double* fetch_ms, double* ffn_ms,
                               double* step_ms) {
  if (!g) return fail(FT_ERR_INVALID_ARG, "null step graph");
  if (!g->timing || !g->launched) return fail(FT_ERR_STATE, "graph was created without timing or never launched");
  const int L = g->L;
  CU(wait_event(g->ev[6 * L + 1]));
  float ms = 0.0f;
  for (int l = 0; l < L; ++l) {
    if (route_ms) {
      CU(cudaEventElapsedTime(&ms, g->ev[2 * l], g->ev[2 * l + 1]));
      route_ms[l] = ms;
    }
    if (ffn_ms) {
      CU(cudaEventElapsedTime(&ms, g->ev[2 * L + 2 * l], g->ev[2 * L + 2 * l + 1]));
      ffn_ms[l] = ms;
    }
    if (fetch_ms) {
      ms = 0.0f;
      if (g->fetch_events) CU(cudaEventElapsedTime(&ms, g->ev[4 * L + 2 * l], g->ev[4 * L + 2 * l + 1]));
      fetch_ms[l] = ms;
    }
  }
  if (step_ms) {
    CU(cudaEventElapsedTime(&ms, g->ev[6 * L], g->ev[6 * L + 1]));
    *step_ms = ms;
  }
  return FT_OK;
}

}  // extern "C"
