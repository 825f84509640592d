/*
 * ft.h - C ABI of libft, the GB300 (sm_103a) hot path of a two-tier MoE
 * expert-offload engine: the full routed-expert bank stays in host memory and
 * one GPU expert cache, shared by every MoE layer and keyed by
 * (layer, expert), holds the experts the FFN reads.
 *
 * Source of the method: "FreeToken: Efficient Edge-Native MoE Serving with
 * Bandwidth-Adaptive Execution" (paper summary page), design paragraph
 * (two-tier expert memory; an elastic expert cache shared by all MoE layers,
 * slots managed by logical (layer, expert) id; routing dedup, hit
 * classification and LRU victim selection in one GPU kernel with no per-layer
 * host sync; cache rebuilt at scheduler safe points when the VRAM budget
 * changes; weights stored in the runtime layout) and ablation paragraph
 * (global LRU; double buffering of expert transfers); "FreeToken: az VRAM ile
 * büyük MoE modelleri", intro (experts in host RAM, an LRU expert cache on the
 * GPU, misses streamed over the host link).
 *
 * Conventions
 * - Every call returns ft_status; FT_OK is 0.  No call throws.  On an error
 *   ft_last_error() returns a message for the calling thread.
 * - Pointers named "device" must point to device memory of the cache's GPU;
 *   "host" pointers to host memory.  The caller owns every buffer it passes;
 *   the library owns what it allocates (tables, plans, scratch, streams,
 *   events) and frees it in ft_cache_destroy.
 * - Stream handles are cudaStream_t values passed as void*.
 * - Calls that enqueue GPU work are asynchronous: they return once the work
 *   is enqueued.  Calls marked "synchronous" wait for the cache's streams.
 * - One host thread drives one ft_cache.  Calls on one cache must not
 *   overlap.
 * - Device-side failures (a capacity shortfall, a bounds check, a bounded
 *   wait that ran out) cannot be reported by the call that enqueued them;
 *   they set a sticky device status that the next synchronous call
 *   (ft_synchronize, ft_get_stats, ...) returns.
 */
#ifndef FT_H_
#define FT_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum ft_status {
  FT_OK = 0,
  FT_ERR_INVALID_ARG = 1, /* bad shape, pointer, layer or size */
  FT_ERR_CUDA = 2,        /* a CUDA runtime call failed; see ft_last_error() */
  FT_ERR_OOM = 3,         /* a library allocation failed */
  FT_ERR_CAPACITY = 4,    /* fewer victim slots than misses (pool too small) */
  FT_ERR_STATE = 5,       /* call out of order (forward before fetch, ...) */
  FT_ERR_TIMEOUT = 6,     /* a bounded wait ran out */
  FT_ERR_CHECKED = 7,     /* a device-side bounds check failed */
  FT_ERR_UNSUPPORTED = 8  /* shape or mode this build does not implement */
} ft_status;

/* Expert weight formats.  The FFN input x is float32 for FT_W_F32 and bf16
 * for the other two; the FFN output y is always float32 (the accumulation
 * precision; the caller rounds it into its residual stream). */
typedef enum ft_wdtype {
  FT_W_F32 = 0,
  FT_W_BF16 = 1,
  FT_W_FP8E4M3_B128 = 2 /* OCP e4m3 weights, one bf16 scale per 128x128 block */
} ft_wdtype;

typedef enum ft_fetch_mode {
  /* cudaMemcpyAsync per miss, issued by a library host thread that reads each
   * event's miss list from a ring the route kernel writes to mapped host
   * memory; the FFN waits for a ready flag set after the copies.  Copy engines
   * leave the SMs and their memory path to the kernels. */
  FT_FETCH_COPY_ENGINE = 0,
  FT_FETCH_SM_PULL = 1 /* a kernel on the copy stream loads the blobs over the host link */
} ft_fetch_mode;

/*
 * Expert blob = the runtime layout of one routed expert, identical in the
 * host bank and in a device slot:
 *   Wg [inter][hidden] | Wu [inter][hidden] | Wd [hidden][inter]
 * row-major, element type per ft_wdtype; for FT_W_FP8E4M3_B128 followed by
 * bf16 scales, one per 128x128 block of each matrix ([out][in] blocks,
 * row-block major) in the order Wg, Wu, Wd.
 * The FFN of expert e on token x is  Wd (silu(Wg x) * (Wu x)).
 */
typedef struct ft_cache_config {
  int32_t num_layers;  /* L: MoE layers sharing the cache */
  int32_t num_experts; /* E: routed experts per layer, 1..1024 */
  int32_t top_k;       /* k: experts per token, 1..min(E, 32) */
  int32_t hidden;      /* H: multiple of 128 (of 8 for FT_W_F32) */
  int32_t inter;       /* I: multiple of 128 (of 8 for FT_W_F32) */
  int32_t wdtype;      /* ft_wdtype */
  const void* host_bank;     /* host: [bank_blobs][expert_bytes].  Best allocated with cudaHostAlloc: on
                                GB300 the GPU reads that several times faster over the host link than
                                memory page-locked later.  Memory that is not pinned yet is registered
                                (cudaHostRegister, mapped) by create and stays registered while any
                                cache of this process uses it. */
  uint64_t host_bank_bytes;  /* >= bank_blobs * expert_bytes */
  int64_t bank_blobs;        /* physical blobs; key (l, e) reads blob (l*E + e) mod bank_blobs.
                                L*E for a full bank; fewer aliases blobs to save host RAM */
  int32_t max_tokens;        /* largest T passed to ft_route_classify / ft_moe_forward */
  int32_t fetch_mode;        /* ft_fetch_mode */
  int32_t pull_ctas;         /* CTAs of the SM-pull fetch kernel; 0 = library default */
  int32_t copy_streams;      /* copy-engine mode: 1 or 2 streams the misses alternate over; 0 = 1 */
  int32_t fetch_warps;       /* SM-pull mode: warps per SM of each FFN kernel that copy the next layer's
                                misses over the host link (1..4); 0 = library default (2) */
} ft_cache_config;

typedef struct ft_cache ft_cache; /* opaque, library-owned */
typedef struct ft_step_graph ft_step_graph; /* opaque, library-owned */

/* Counters accumulated since create (or the last ft_reset_stats). */
typedef struct ft_stats {
  int64_t events;          /* layer events classified */
  int64_t unique_experts;  /* sum over events of |U| */
  int64_t hits;            /* sum of |H| */
  int64_t misses;          /* sum of |M| */
  int64_t evictions;       /* misses that replaced an occupied slot, plus resize drops */
  int64_t bytes_fetched;   /* misses * expert_bytes */
  int64_t kernel_launches; /* kernels this library launched */
  int64_t memcpy_calls;    /* cudaMemcpyAsync calls issued for misses */
} ft_stats;

/* Per-phase GPU time from CUDA events recorded around the library's own
 * launches (enabled by ft_timing_enable); milliseconds and counts. */
typedef struct ft_timing {
  double route_ms;  int64_t route_n;   /* route_classify kernel, compute stream */
  double fetch_ms;  int64_t fetch_n;   /* miss copies, copy stream (first to last copy of a layer) */
  double ffn_ms;    int64_t ffn_n;     /* expert FFN kernels of one ft_moe_forward, compute stream */
  double gemm1_ms;  int64_t gemm1_n;   /* prefill forwards: the gate/up + SwiGLU tensor-core GEMM alone */
  double gemm2_ms;  int64_t gemm2_n;   /* prefill forwards: the down tensor-core GEMM alone */
} ft_timing;

/* Header of one layer's plan (see ft_get_plan). */
typedef struct ft_plan_info {
  int32_t event;     /* event number t of the classification */
  int32_t n_tokens;  /* T */
  int32_t n_unique;  /* |U| */
  int32_t n_miss;    /* |M| */
} ft_plan_info;

/* Bytes of one expert blob; 0 for an unsupported shape. */
size_t ft_expert_bytes(int32_t hidden, int32_t inter, int32_t wdtype);

/*
 * The host tier: pinned, device-mapped host memory of exactly `bytes` bytes
 * for an expert bank ("FreeToken: az VRAM ile büyük MoE modelleri", intro:
 * the experts that do not fit stay in host RAM and are streamed from it),
 * portable across the process's contexts, content undefined.  The caller owns
 * it and frees it with ft_host_bank_free after the last cache that uses it is
 * destroyed.  Errors: FT_ERR_INVALID_ARG (bytes 0, null out), FT_ERR_OOM
 * (*host is then NULL).  ft_host_bank_free(NULL) does nothing; FT_ERR_CUDA if
 * the runtime refuses the pointer.
 */
ft_status ft_host_bank_alloc(uint64_t bytes, void** host);
ft_status ft_host_bank_free(void* host);

/*
 * Budget-driven sizing (the "automatic" cache size of the pages' runtime:
 * "FreeToken vs vLLM on one RTX 3090", Runtime configurations; the cache is
 * rebuilt when the VRAM budget changes: "FreeToken: Efficient Edge-Native MoE
 * Serving ...", design paragraph).  No GPU work; usable before any device is
 * touched.
 *
 * ft_cache_overhead_bytes: device bytes ft_cache_create allocates for a cache
 * of `num_slots` slots with this configuration (slot tables, LRU log, plans,
 * scratch, prefill buffers; each allocation rounded to 512 bytes), not
 * counting the caller's slot pool.  0 for an invalid configuration.
 *
 * ft_slots_for_budget: the most slots C with C * expert_bytes plus the
 * overhead of C slots within `budget_bytes` (a caller derives the budget from
 * the free device memory minus what it keeps for everything else, and again
 * when that changes; ft_cache_resize then moves the cache to the new size at a
 * safe point).  Errors: FT_ERR_INVALID_ARG (configuration), FT_ERR_CAPACITY
 * (the budget holds fewer slots than 2 * min(max_tokens * top_k,
 * num_experts); *num_slots is 0).
 */
uint64_t ft_cache_overhead_bytes(const ft_cache_config* cfg, int64_t num_slots);
ft_status ft_slots_for_budget(const ft_cache_config* cfg, uint64_t budget_bytes, int64_t* num_slots);

/*
 * Create a cache over `num_slots` slots of the caller's device pool
 * `slot_pool` ([num_slots][expert_bytes], device, 256-byte aligned, owned by
 * the caller and valid until destroy or the next resize).  The cache starts
 * empty.  `compute_stream` (cudaStream_t, may be NULL for the legacy default
 * stream) receives the routing and FFN kernels; the library creates its own
 * copy stream(s).  Registers the host bank with CUDA if it is not pinned
 * (and unregisters it on destroy).  Synchronous.
 * Errors: FT_ERR_INVALID_ARG (shapes, null pointers, bank too small,
 * expert_bytes not a multiple of 16), FT_ERR_CAPACITY when num_slots <
 * 2 * min(max_tokens * top_k, num_experts) (the pool could not hold one
 * event's experts plus the previous event's pinned ones), FT_ERR_OOM,
 * FT_ERR_CUDA.
 */
ft_status ft_cache_create(const ft_cache_config* cfg, void* slot_pool, int64_t num_slots, void* compute_stream,
                          ft_cache** out);

/* Destroy a cache: waits for its streams, frees library memory.  NULL is a
 * no-op. */
ft_status ft_cache_destroy(ft_cache* cache);

/*
 * Resize the cache at a safe point ("rebuilt at scheduler safe points when
 * the VRAM budget changes").  Synchronous: waits for both streams first.
 * Keeps the min(occupied, new_num_slots) entries that LRU would evict last;
 * survivors in slots < new_num_slots stay put, the others move (in ascending
 * old-slot order) to the lowest free slots; last-use times are kept.  When
 * `new_pool` differs from the current pool every survivor is copied into it
 * (the old pool must stay valid until the call returns); when it is the same
 * pointer, blobs move in place.  The first event after a resize pins nothing.
 * Errors: FT_ERR_INVALID_ARG, FT_ERR_CAPACITY (same bound as create),
 * FT_ERR_STATE (a fetch is still pending), FT_ERR_CUDA, FT_ERR_OOM.
 */
ft_status ft_cache_resize(ft_cache* cache, void* new_pool, int64_t new_num_slots);

/*
 * Route one layer's token batch and update the cache, in one kernel: top-k
 * + gates per token, dedup of the batch's experts,
 * hit/miss classification, global-LRU victims for the misses, table update.
 *   logits   device, float32 [T][E], row-major
 *   topk_idx device, int32 [T][k] or NULL: experts per token in selection
 *            order (logit descending, lower index first on ties)
 *   topk_w   device, float32 [T][k] or NULL: softmax over the k selected logits
 * The event number t increments by one per call.  Victims are the least
 * recently used slots excluding this event's hits and the previous event's
 * slots (which the previous layer's FFN may still read).  T may be 0.
 * The kernel runs on a library stream that first waits for all work already
 * enqueued on the compute stream (the logits, and the FFN of two layers back
 * in the double-buffered schedule); its outputs are ordered before this
 * layer's ft_moe_forward on the compute stream and before ft_synchronize,
 * not before other work the caller enqueues in between.
 * Errors: FT_ERR_INVALID_ARG (layer, T > max_tokens, null logits),
 * FT_ERR_STATE (this layer's previous plan is still being fetched and its
 * fetch failed), FT_ERR_UNSUPPORTED (T > 8 in copy-engine mode: the prefill
 * kernels read the slots without waiting for the copy thread), FT_ERR_CUDA.
 */
ft_status ft_route_classify(ft_cache* cache, int32_t layer, const float* logits, int32_t T, int32_t* topk_idx,
                            float* topk_w);

/*
 * Copy the layer's misses (from its last ft_route_classify) from the host
 * bank into their victim slots, after the classification completes and
 * after the FFN of two events before (whose slots may be the victims).
 * Asynchronous; the compute stream does not wait here, so the next layer's
 * misses stream while this layer computes.  SM-pull mode: the copy is
 * deferred and done by the copy warps of the next ft_moe_forward of another
 * layer (one kernel per layer moves the next layer's experts over the host
 * link while this layer's stream from HBM); a forward of the layer itself,
 * a prefill forward or any synchronising call runs it as a pull kernel on the
 * copy stream instead.  Copy-engine mode: the library's copy thread issues one
 * cudaMemcpyAsync per miss on the copy stream.
 * Errors: FT_ERR_INVALID_ARG, FT_ERR_STATE (no classification pending for
 * this layer), FT_ERR_CUDA.
 */
ft_status ft_fetch_misses(ft_cache* cache, int32_t layer);

/*
 * The layer's MoE FFN on the compute stream, reading expert weights from the
 * cache slots:  y[t] = sum_j topk_w[t][j] * Wd h,  h = silu(Wg x[t]) * (Wu x[t]).
 *   x  device [T][H]: float32 for FT_W_F32, bf16 otherwise
 *   y  device [T][H]: float32; fully overwritten
 * T must equal the T of the layer's last ft_route_classify.  The compute
 * stream first waits for the layer's fetch.  T <= 8 (decode) runs one fused
 * kernel per layer (gate/up, SwiGLU, down and the combine, adding into y in
 * no fixed order, so y is reproducible to fp32 rounding; in SM-pull mode it
 * also copies the next requested layer's misses), launched as a programmatic
 * dependent of the kernel before it on the stream.  Larger T (prefill; bf16
 * or fp8 weights, hidden and inter multiples of 128) groups the rows by
 * expert and runs the gate/up + SwiGLU and down projections as grouped
 * tensor-core GEMMs (fp8 weights dequantised to fp16 with their block scales
 * on the way), then combines each token's picks in pick order.
 * Errors: FT_ERR_INVALID_ARG, FT_ERR_STATE (no fetch issued for the layer's
 * current plan), FT_ERR_UNSUPPORTED (a prefill T with other weight types or
 * shapes, or a cache created with max_tokens <= 8), FT_ERR_CUDA.
 */
ft_status ft_moe_forward(ft_cache* cache, int32_t layer, const void* x, int32_t T, void* y);

/* Wait for the compute and copy streams; returns the sticky device status
 * (FT_ERR_CAPACITY, FT_ERR_CHECKED, FT_ERR_TIMEOUT) if one was raised.
 * Synchronous. */
ft_status ft_synchronize(ft_cache* cache);

/*
 * Copy a layer's current plan to host (synchronous; test and debug use).
 * Any array pointer may be NULL.  Host arrays must hold num_experts entries.
 *   unique_expert  ascending experts of U        unique_slot  slot of each after the event
 *   hit            1 = hit, 0 = miss             miss_expert  ascending misses
 *   miss_slot      victim slot of each miss      evicted_key  key (l*E+e) the victim held, -1 if empty
 */
ft_status ft_get_plan(ft_cache* cache, int32_t layer, ft_plan_info* info, int32_t* unique_expert,
                      int32_t* unique_slot, uint8_t* hit, int32_t* miss_expert, int32_t* miss_slot,
                      int32_t* evicted_key);

/* Copy the slot tables to host (synchronous).  key_to_slot: [L*E] (-1 =
 * absent); slot_key, slot_ts: [num_slots] (-1 = empty / never used).  Any
 * pointer may be NULL. */
ft_status ft_get_tables(ft_cache* cache, int32_t* key_to_slot, int32_t* slot_key, int32_t* slot_ts);

/* Counters (synchronous). */
ft_status ft_get_stats(ft_cache* cache, ft_stats* out);
ft_status ft_reset_stats(ft_cache* cache);

/* Current number of slots and pool pointer. */
ft_status ft_get_pool(ft_cache* cache, void** pool, int64_t* num_slots);

/* The copy stream (cudaStream_t as void*) the miss copies run on (the
 * first one when copy_streams is 2). */
ft_status ft_get_copy_stream(ft_cache* cache, void** stream);

/* Test and debug knob, copy-engine mode only: while `paused` is 1 the
 * library's copy thread serves no event, so FFN kernels that wait for a
 * layer's copies run into their bounded wait (about one second), record
 * FT_ERR_TIMEOUT and finish; the next synchronous call reports it.  Setting 0
 * lets the thread continue where it stopped.  Errors: FT_ERR_INVALID_ARG,
 * FT_ERR_STATE (SM-pull cache: no copy thread). */
ft_status ft_debug_pause_copies(ft_cache* cache, int32_t paused);

/* 1 if this library is the bounds-checked build (compiled with -DFT_CHECKED:
 * every kernel checks the table and plan indices it dereferences; one out of
 * range raises FT_ERR_CHECKED in the sticky device status, which the next
 * synchronous call returns, and the access is skipped instead of made), else
 * 0. */
int32_t ft_checked_build(void);

/* Test knob of the bounds-checked build: after the cache's work so far,
 * overwrite the slot table entry of key (layer * E + expert) with `slot`, so
 * that a test can hand the kernels an index out of range.  Errors:
 * FT_ERR_INVALID_ARG (null cache, key outside [0, L*E)), FT_ERR_STATE (a
 * build without the checks, whose kernels would read such a table out of
 * range). */
ft_status ft_debug_set_key_slot(ft_cache* cache, int32_t key, int32_t slot);

/* Enable (1) or disable (0) per-phase CUDA-event timing; enabling clears the
 * totals and creates the events up front (no timed phase pays for creating
 * them).  ft_get_timing waits for the streams and returns the totals.
 * Errors: FT_ERR_INVALID_ARG (null cache), FT_ERR_CUDA (events could not be
 * created), or an error the synchronisation reports. */
ft_status ft_timing_enable(ft_cache* cache, int32_t on);
ft_status ft_get_timing(ft_cache* cache, ft_timing* out);

/*
 * Decode expert FFN that allocates nothing (no counterpart in the paper: an
 * addition for callers that cannot allocate device memory, such as an engine
 * whose memory planner owns all device memory, or a serving loop where a
 * cudaMalloc/cudaFree stall is not acceptable; ft_moe_forward needs a cache,
 * and ft_cache_create allocates).  Same result as ft_moe_forward's decode path
 * for the same weights and routing:
 *   y[t] = sum_j topk_w[t][j] * Wd h,  h = silu(Wg x[t]) * (Wu x[t]),
 * with expert e's blob read from slot expert_slot[e] of slot_pool.
 *   slot_pool    device [num_slots][expert_bytes] expert blobs (layout above)
 *   expert_slot  device int32 [num_experts]: slot of each expert; a pick whose
 *                expert id or slot is out of range contributes nothing
 *   topk_idx     device int32 [T][top_k], distinct experts within a row;
 *                topk_w device float32 [T][top_k]
 *   x            device [T][hidden], float32 for FT_W_F32 else bf16
 *   y            device [T][hidden] float32
 *   stream       cudaStream_t (void*), NULL = legacy default stream
 * Asynchronous on `stream`.  Working memory is one static 1 MiB device array
 * per GPU.  With lazy module loading (the CUDA default) it is reserved on a
 * GPU at the first call there, where a failure to reserve it is reported, and
 * kept until the process exits (with CUDA_MODULE_LOADING=EAGER it is reserved
 * when the library loads).  A caller whose memory planner then takes all
 * device memory should make one warm-up call first.  That first call on a
 * device (and the first after the current context changes) also looks up the
 * array's address: make it before any stream capture.  Limits: T <= 8,
 * hidden % 8 == 0, and T*top_k*inter*4 bytes of intermediate within 1,032,192
 * bytes (T*top_k <= 64 at inter 4096); other sizes return FT_ERR_INVALID_ARG
 * with a message, before any GPU work.  All calls share the array: calls whose
 * kernels overlap on the GPU (other streams or threads) race.  A bounded wait
 * that runs out inside the kernels leaves y incomplete and sets a sticky
 * status word in the array; read it with ft_moe_decode_ffn_static_status.
 */
ft_status ft_moe_decode_ffn_static(int32_t hidden, int32_t inter, int32_t wdtype, int32_t num_experts,
                                   int32_t top_k, const void* slot_pool, int64_t num_slots,
                                   const int32_t* expert_slot, const int32_t* topk_idx, const float* topk_w,
                                   const void* x, int32_t T, void* y, void* stream);

/* Status of the static-scratch FFN calls on the current device: waits for
 * `stream` (cudaStream_t as void*, NULL = legacy default stream), then returns
 * FT_ERR_TIMEOUT if a kernel of an earlier ft_moe_decode_ffn_static call gave
 * up a bounded wait (its y is incomplete), else FT_OK.  Reading clears the
 * word.  Allocates nothing.  Synchronous. */
ft_status ft_moe_decode_ffn_static_status(void* stream);

/*
 * Step graphs: one decode/prefill step of all L layers captured into a CUDA
 * graph, so a step costs one launch instead of ~5 API calls per layer (the
 * pages capture their whole execution layer in a CUDA graph: "FreeToken:
 * Efficient Edge-Native MoE Serving ...", design paragraph).  The captured
 * schedule is the one ft_route_classify / ft_fetch_misses / ft_moe_forward
 * give when called as
 *   double_buffer: route(0); fetch(0); for l: { route(l+1); fetch(l+1); forward(l) }
 *   serial:        for l: { route(l); fetch(l); forward(l) }
 * with logits[l] (device f32 [T][E]), x[l] (device [T][H]) and y[l] (device
 * f32 [T][H]) baked in: refill those buffers before each launch.  The event
 * counter and the pin rule advance on the device, so replays continue the
 * cache's decision stream exactly as direct calls would.  Works in both fetch
 * modes (in copy-engine mode the library's copy thread serves the replays'
 * events from the ring as they are routed).  Needs no layer with a fetched,
 * not yet forwarded plan (FT_ERR_STATE).  Create is synchronous; launch
 * enqueues the step on the cache's compute stream.  In copy-engine mode a
 * launch first waits (polling, no blocking runtime call) for the end of the
 * launch two before it, so at most two steps are queued: the FFNs wait for
 * the library's copy thread, which must never be stuck behind a host thread
 * blocked in a full launch queue.  In SM-pull mode the routing of every layer
 * runs ahead of the FFNs from the step's start (the logits are graph inputs)
 * and each layer's pull kernel waits for the FFN of two events before.  With `timing` set the
 * graph records events around each layer's route kernel, miss fetch and FFN
 * kernels; ft_step_graph_timing waits for the last launch and returns them
 * (ms; any pointer may be NULL; arrays hold L entries).  In copy-engine mode
 * the misses are copied by the library's copy thread outside the graph, so
 * the graph has no fetch events: fetch_ms is 0 there (ft_timing_enable /
 * ft_get_timing time those copies instead).
 */
ft_status ft_step_graph_create(ft_cache* cache, const float* const* logits, const void* const* x, float* const* y,
                               int32_t T, int32_t double_buffer, int32_t timing, ft_step_graph** out);
ft_status ft_step_graph_launch(ft_step_graph* graph);
ft_status ft_step_graph_timing(ft_step_graph* graph, double* route_ms, double* fetch_ms, double* ffn_ms,
                               double* step_ms);
/* Timeline of the graph's last launch (waits for it): t_ms[6*l + j] = time
 * from the step's start to the route begin/end (j = 0, 1), fetch begin/end
 * (2, 3) and FFN begin/end (4, 5) of layer l.  Needs a timing graph.  The
 * fetch entries are -1 in copy-engine mode (no fetch events in the graph). */
ft_status ft_step_graph_trace(ft_step_graph* graph, double* t_ms);
ft_status ft_step_graph_destroy(ft_step_graph* graph);

const char* ft_status_str(ft_status s);
/* Message of the calling thread's last error ("" if none). */
const char* ft_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* FT_H_ */
