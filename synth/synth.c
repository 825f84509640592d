/*
 * Seeded synthetic input generators, shared by the CPU oracle and by the CUDA
 * path's tests and benchmark.  Nothing here computes any step of the MoE
 * expert-cache method: this file only makes inputs (router logits, hidden
 * states, expert weight blobs).  Random numbers come from one counter-based
 * generator, SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014): the n-th draw of stream `key` is the
 * SplitMix64 finaliser applied to key + (n+1)*gamma.  Normal draws use the
 * Box-Muller transform on pairs of uniforms.
 *
 * Compiled as a plain shared library (gcc, -ffp-contract=off) and called from
 * Python through ctypes.  All bulk routines split their work over pthreads;
 * the output never depends on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define SM_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t sm_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

/* n-th output of the SplitMix64 stream whose state starts at `key`. */
static inline uint64_t sm_at(uint64_t key, uint64_t n) { return sm_mix(key + (n + 1) * SM_GAMMA); }

/* Stream key from a seed and four coordinates (stream id, and up to three indices). */
uint64_t synth_key(uint64_t seed, uint64_t a, uint64_t b, uint64_t c, uint64_t d) {
  uint64_t h = sm_mix(seed + SM_GAMMA);
  h = sm_mix(h ^ sm_mix(a + 1 * SM_GAMMA));
  h = sm_mix(h ^ sm_mix(b + 2 * SM_GAMMA));
  h = sm_mix(h ^ sm_mix(c + 3 * SM_GAMMA));
  h = sm_mix(h ^ sm_mix(d + 4 * SM_GAMMA));
  return h;
}

uint64_t synth_u64(uint64_t key, uint64_t n) { return sm_at(key, n); }

/* Uniform in the open interval (0, 1) from the top 24 bits of draw n. */
static inline float unif24(uint64_t key, uint64_t n) {
  return ((float)(sm_at(key, n) >> 40) + 0.5f) * (1.0f / 16777216.0f);
}

/* Uniform in (0, 1) from the top 53 bits of draw n (double). */
static inline double unif53(uint64_t key, uint64_t n) {
  return ((double)(sm_at(key, n) >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}

/* Standard normal number i of stream `key`: Box-Muller on draws 2*(i/2) and
 * 2*(i/2)+1; even i takes the cosine branch, odd i the sine branch. */
static inline float normal_at(uint64_t key, uint64_t i) {
  uint64_t p = i >> 1;
  float u1 = unif24(key, 2 * p), u2 = unif24(key, 2 * p + 1);
  float r = sqrtf(-2.0f * logf(u1));
  float th = 6.28318530717958647692f * u2;
  return (i & 1) ? r * sinf(th) : r * cosf(th);
}

/* Both normals of pair p (elements 2p and 2p+1), same values as normal_at. */
static inline void normal_pair(uint64_t key, uint64_t p, float* z0, float* z1) {
  float u1 = unif24(key, 2 * p), u2 = unif24(key, 2 * p + 1);
  float r = sqrtf(-2.0f * logf(u1));
  float th = 6.28318530717958647692f * u2;
  *z0 = r * cosf(th);
  *z1 = r * sinf(th);
}

/* out[i] = scale * N_(start+i), i < n, computed pairwise. */
static void normal_span(uint64_t key, uint64_t start, int64_t n, float scale, float* out) {
  int64_t i = 0;
  if ((start & 1) && n > 0) { out[0] = scale * normal_at(key, start); i = 1; }
  for (; i + 1 < n; i += 2) {
    float a, b;
    normal_pair(key, (start + (uint64_t)i) >> 1, &a, &b);
    out[i] = scale * a;
    out[i + 1] = scale * b;
  }
  if (i < n) out[i] = scale * normal_at(key, start + (uint64_t)i);
}

/* ---- conversions (input encoding only) --------------------------------- */

/* fp32 -> bf16 bits, round to nearest even (finite inputs). */
static inline uint16_t f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}
static inline float bf16_to_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* fp32 -> OCP FP8 E4M3 (bias 7, max 448, no infinities), round to nearest
 * even, saturating to +-448.  Used only to encode generated weights. */
static uint8_t f32_to_e4m3_sat(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  uint8_t sign = (uint8_t)((u >> 24) & 0x80);
  uint32_t a = u & 0x7FFFFFFFu;
  if (a > 0x7F800000u) return 0x7F;          /* NaN: never produced by the generators */
  if (a >= 0x43E00000u) return sign | 0x7E;  /* |f| >= 448 saturates */
  int ue = (int)(a >> 23) - 127;
  if (ue < -6) {                             /* e4m3 subnormal range: multiples of 2^-9 */
    float af;
    memcpy(&af, &a, 4);
    int m = (int)rintf(af * 512.0f);         /* exact scaling, then round to nearest even */
    return sign | (uint8_t)m;                /* m == 8 is the smallest normal, code 0x08 */
  }
  uint32_t q = a >> 20;                      /* exponent and top 3 fraction bits */
  uint32_t rest = a & 0xFFFFFu, half = 0x80000u;
  if (rest > half || (rest == half && (q & 1u))) q += 1; /* carries into the exponent */
  int e = (int)(q >> 3) - 127;
  uint32_t m = q & 7u;
  if (e > 8 || (e == 8 && m > 6)) return sign | 0x7E;
  return sign | (uint8_t)(((e + 7) << 3) | (int)m);
}

uint8_t synth_e4m3_encode(float f) { return f32_to_e4m3_sat(f); }
uint16_t synth_bf16_encode(float f) { return f32_to_bf16(f); }

void synth_f32_to_bf16(const float* in, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = f32_to_bf16(in[i]);
}
void synth_bf16_to_f32(const uint16_t* in, float* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = bf16_to_f32(in[i]);
}

/* ---- threading helper --------------------------------------------------- */

typedef void (*range_fn)(void* ctx, int64_t lo, int64_t hi);
typedef struct { range_fn fn; void* ctx; int64_t lo, hi; } range_job;
static void* range_thread(void* p) {
  range_job* j = (range_job*)p;
  j->fn(j->ctx, j->lo, j->hi);
  return NULL;
}
/* Runs fn over [0, n) split into `threads` ranges; below `min_items` items
 * the call stays on the calling thread (thread start-up would dominate). */
static void parallel_for(range_fn fn, void* ctx, int64_t n, int threads, int64_t min_items) {
  if (threads < 1) threads = 1;
  if (threads > 256) threads = 256;
  if (n < min_items || n < 2 || threads == 1) { fn(ctx, 0, n); return; }
  if (threads > n) threads = (int)n;
  pthread_t tid[256];
  range_job jobs[256];
  for (int t = 0; t < threads; ++t) {
    jobs[t].fn = fn; jobs[t].ctx = ctx;
    jobs[t].lo = n * t / threads; jobs[t].hi = n * (t + 1) / threads;
    if (pthread_create(&tid[t], NULL, range_thread, &jobs[t]) != 0) {
      range_thread(&jobs[t]);
      tid[t] = 0;
    }
  }
  for (int t = 0; t < threads; ++t)
    if (tid[t]) pthread_join(tid[t], NULL);
}

/* ---- normal arrays ------------------------------------------------------ */

typedef struct { uint64_t key; uint64_t start; float scale; float* out; } normal_ctx;
static void normal_range(void* p, int64_t lo, int64_t hi) {
  normal_ctx* c = (normal_ctx*)p;
  normal_span(c->key, c->start + (uint64_t)lo, hi - lo, c->scale, c->out + lo);
}
/* out[i] = scale * N_(start+i) of stream `key` */
void synth_normal_f32(uint64_t key, uint64_t start, int64_t n, float scale, float* out, int threads) {
  normal_ctx c = {key, start, scale, out};
  parallel_for(normal_range, &c, n, threads, 1 << 16);
}

/* ---- expert weight blobs ------------------------------------------------ */
/*
 * Blob layout (the runtime layout of one routed expert, shared by the host
 * bank and the device slots):  Wg[I][H] | Wu[I][H] | Wd[H][I], row-major,
 * element type f32, bf16 or fp8-e4m3; for fp8 the three matrices are followed
 * by bf16 block scales, one per 128x128 block of each matrix in the order
 * Wg (I/128 x H/128), Wu (I/128 x H/128), Wd (H/128 x I/128), row-block major.
 * Element n of the blob (counted over the three matrices, row-major) is
 * weight_at(key, n): an Irwin-Hall(4) approximation of N(0, 0.02^2) taken
 * from one SplitMix64 draw (integer sum of its four 16-bit fields, centred,
 * times one float constant), so a 64 GB bank takes seconds, not minutes.
 */
enum { W_F32 = 0, W_BF16 = 1, W_FP8 = 2 };

/* sum of four 16-bit uniforms has variance (65536^2 - 1)/3, sd ~ 37837.23 */
#define WEIGHT_SCALE (0.02f / 37837.2265f)
static inline float weight_at(uint64_t key, uint64_t n) {
  uint64_t r = sm_at(key, n);
  int32_t s = (int32_t)(r & 0xFFFF) + (int32_t)((r >> 16) & 0xFFFF) + (int32_t)((r >> 32) & 0xFFFF) +
              (int32_t)(r >> 48);
  return (float)(s - 131070) * WEIGHT_SCALE;
}
static void weight_span(uint64_t key, uint64_t start, int64_t n, float* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = weight_at(key, start + (uint64_t)i);
}

int64_t synth_expert_bytes(int hidden, int inter, int wdtype) {
  int64_t n = 3LL * hidden * inter;
  if (wdtype == W_F32) return 4 * n;
  if (wdtype == W_BF16) return 2 * n;
  if (wdtype == W_FP8) {
    if (hidden % 128 || inter % 128) return -1;
    return n + 2LL * 3 * (hidden / 128) * (inter / 128);
  }
  return -1;
}

typedef struct {
  uint64_t seed; int hidden, inter, wdtype; const int64_t* blob_ids; uint8_t* out; int64_t eb;
} bank_ctx;

static void gen_blob(const bank_ctx* c, int64_t blob_id, uint8_t* dst) {
  const int H = c->hidden, I = c->inter;
  const uint64_t key = synth_key(c->seed, 0x57E1, (uint64_t)blob_id, 0, 0);
  const int64_t n = 3LL * H * I;
  if (c->wdtype == W_F32) {
    weight_span(key, 0, n, (float*)dst);
  } else if (c->wdtype == W_BF16) {
    uint16_t* w = (uint16_t*)dst;
    for (int64_t i = 0; i < n; ++i) w[i] = f32_to_bf16(weight_at(key, (uint64_t)i));
  } else {
    uint8_t* q = dst;
    uint16_t* scales = (uint16_t*)(dst + n);
    int64_t si = 0;
    float blk[128 * 128];
    for (int mat = 0; mat < 3; ++mat) {
      const int rows = mat < 2 ? I : H, cols = mat < 2 ? H : I;
      const int64_t base = (int64_t)mat * H * I;
      for (int rb = 0; rb < rows / 128; ++rb)
        for (int cb = 0; cb < cols / 128; ++cb) {
          float amax = 0.0f;
          for (int r = 0; r < 128; ++r) {
            int64_t e0 = base + (int64_t)(rb * 128 + r) * cols + cb * 128;
            weight_span(key, (uint64_t)e0, 128, blk + r * 128);
            for (int cc = 0; cc < 128; ++cc) {
              float a = fabsf(blk[r * 128 + cc]);
              if (a > amax) amax = a;
            }
          }
          uint16_t sb = f32_to_bf16(amax / 448.0f);
          float s = bf16_to_f32(sb);
          scales[si++] = sb;
          for (int r = 0; r < 128; ++r)
            for (int cc = 0; cc < 128; ++cc) {
              int64_t e = base + (int64_t)(rb * 128 + r) * cols + cb * 128 + cc;
              q[e] = s > 0.0f ? f32_to_e4m3_sat(blk[r * 128 + cc] / s) : 0;
            }
        }
    }
  }
}

static void bank_range(void* p, int64_t lo, int64_t hi) {
  bank_ctx* c = (bank_ctx*)p;
  for (int64_t b = lo; b < hi; ++b) gen_blob(c, c->blob_ids[b], c->out + b * c->eb);
}

/* Writes n_blobs consecutive expert blobs (blob_ids[i] -> out + i*expert_bytes). */
int synth_expert_blobs(uint64_t seed, int hidden, int inter, int wdtype, const int64_t* blob_ids,
                       int64_t n_blobs, uint8_t* out, int threads) {
  int64_t eb = synth_expert_bytes(hidden, inter, wdtype);
  if (eb <= 0) return -1;
  bank_ctx c = {seed, hidden, inter, wdtype, blob_ids, out, eb};
  parallel_for(bank_range, &c, n_blobs, threads, 2);
  return 0;
}

/* ---- router logits ------------------------------------------------------ */

/* Zipf(a) routing bias of one layer: a seeded permutation gives expert e the
 * popularity rank r(e) in 1..E; bias_e = log(r^-a / sum_r' r'^-a). */
void synth_zipf_bias(uint64_t seed, int layer, int E, double a, float* bias) {
  uint64_t key = synth_key(seed, 0x21FF, (uint64_t)layer, 0, 0);
  int* perm = (int*)malloc(sizeof(int) * E);
  for (int i = 0; i < E; ++i) perm[i] = i;
  for (int i = E - 1; i > 0; --i) { /* Fisher-Yates */
    int j = (int)(unif53(key, (uint64_t)i) * (double)(i + 1));
    if (j > i) j = i;
    int t = perm[i]; perm[i] = perm[j]; perm[j] = t;
  }
  double z = 0.0;
  for (int r = 1; r <= E; ++r) z += pow((double)r, -a);
  for (int r = 1; r <= E; ++r) bias[perm[r - 1]] = (float)log(pow((double)r, -a) / z);
  free(perm);
}

/*
 * Correlated decode routing of one stream, all steps and layers:
 * out[step][layer][E].  Step 0: logits = N(0,1) + bias.  Step s > 0: keep
 * m ~ Binomial(k, p_keep) experts picked uniformly from the stream's previous
 * chosen set at that layer, draw k-m more without replacement from
 * softmax(N(0,1) + bias) over the others (Gumbel-top-k), and add `lift` to the
 * k chosen logits so they are the top-k by a margin larger than the spread of
 * the rest.  When p_keep < 0 every step is i.i.d. N(0,1) + bias (no lift).
 * When zipf_a <= 0 the bias is zero.
 */
void synth_router_decode(uint64_t seed, int stream, int L, int E, int k, int steps, double zipf_a,
                         double p_keep, float lift, float* out) {
  float* bias = (float*)calloc((size_t)E * L, sizeof(float));
  if (zipf_a > 0)
    for (int l = 0; l < L; ++l) synth_zipf_bias(seed, l, E, zipf_a, bias + (size_t)l * E);
  int* prev = (int*)malloc(sizeof(int) * (size_t)L * k);
  int* cur = (int*)malloc(sizeof(int) * k);
  uint8_t* taken = (uint8_t*)malloc(E);
  double* gkey = (double*)malloc(sizeof(double) * E);
  for (int s = 0; s < steps; ++s)
    for (int l = 0; l < L; ++l) {
      float* row = out + ((size_t)s * L + l) * E;
      const float* b = bias + (size_t)l * E;
      uint64_t kz = synth_key(seed, 0x1061, (uint64_t)stream, (uint64_t)s, (uint64_t)l);
      for (int e = 0; e < E; ++e) row[e] = normal_at(kz, (uint64_t)e) + b[e];
      if (p_keep < 0 || lift == 0.0f) continue;
      uint64_t kc = synth_key(seed, 0xC401, (uint64_t)stream, (uint64_t)s, (uint64_t)l);
      uint64_t draw = 0;
      memset(taken, 0, E);
      int nc = 0;
      if (s > 0) {
        int m = 0;
        for (int j = 0; j < k; ++j) m += unif53(kc, draw++) < p_keep;
        /* uniform m-subset of prev: order prev by random keys, keep first m */
        double rk[64];
        int ord[64];
        for (int j = 0; j < k; ++j) { rk[j] = unif53(kc, draw++); ord[j] = j; }
        for (int a = 1; a < k; ++a) { /* insertion sort by key */
          int o = ord[a];
          int bpos = a - 1;
          while (bpos >= 0 && rk[ord[bpos]] > rk[o]) { ord[bpos + 1] = ord[bpos]; --bpos; }
          ord[bpos + 1] = o;
        }
        for (int j = 0; j < m; ++j) { int e = prev[(size_t)l * k + ord[j]]; cur[nc++] = e; taken[e] = 1; }
      }
      /* Gumbel-top-(k-nc) over the experts not yet taken */
      for (int e = 0; e < E; ++e) {
        double u = unif53(kc, 1000 + (uint64_t)e);
        gkey[e] = taken[e] ? -INFINITY : (double)row[e] - log(-log(u));
      }
      while (nc < k) {
        int best = -1;
        for (int e = 0; e < E; ++e)
          if (!taken[e] && (best < 0 || gkey[e] > gkey[best])) best = e;
        taken[best] = 1;
        cur[nc++] = best;
      }
      for (int j = 0; j < k; ++j) { row[cur[j]] += lift; prev[(size_t)l * k + j] = cur[j]; }
    }
  free(bias); free(prev); free(cur); free(taken); free(gkey);
}

/* Prefill routing of one chunk at one layer: out[T][E] = N(0,1) + bias, i.i.d. per token. */
typedef struct { uint64_t key; int E; const float* bias; float* out; } iid_ctx;
static void iid_range(void* p, int64_t lo, int64_t hi) {
  iid_ctx* c = (iid_ctx*)p;
  for (int64_t i = lo; i < hi; ++i) {
    int e = (int)(i % c->E);
    c->out[i] = normal_at(c->key, (uint64_t)i) + (c->bias ? c->bias[e] : 0.0f);
  }
}
void synth_router_iid(uint64_t seed, int stream, int layer, int T, int E, double zipf_a, float* out, int threads) {
  float* bias = NULL;
  if (zipf_a > 0) {
    bias = (float*)malloc(sizeof(float) * E);
    synth_zipf_bias(seed, layer, E, zipf_a, bias);
  }
  iid_ctx c = {synth_key(seed, 0x11D0, (uint64_t)stream, (uint64_t)layer, 0), E, bias, out};
  parallel_for(iid_range, &c, (int64_t)T * E, threads, 1 << 16);
  free(bias);
}

/* Tie-heavy logits for stress tests: N(0,1) rounded to multiples of 0.25. */
void synth_router_ties(uint64_t seed, int stream, int64_t n, float* out) {
  uint64_t key = synth_key(seed, 0x7133, (uint64_t)stream, 0, 0);
  for (int64_t i = 0; i < n; ++i) out[i] = roundf(4.0f * normal_at(key, (uint64_t)i)) * 0.25f;
}

/* Hidden states: out[T][H] = N(0,1), optionally rounded to bf16 values. */
void synth_hidden(uint64_t seed, int stream, int step, int layer, int T, int H, int round_bf16, float* out,
                  int threads) {
  uint64_t key = synth_key(seed, 0x4AD0, (uint64_t)stream, (uint64_t)step, (uint64_t)layer);
  normal_ctx c = {key, 0, 1.0f, out};
  parallel_for(normal_range, &c, (int64_t)T * H, threads, 1 << 16);
  if (round_bf16)
    for (int64_t i = 0; i < (int64_t)T * H; ++i) out[i] = bf16_to_f32(f32_to_bf16(out[i]));
}
