/*
 * Seeded synthetic inputs for split-tier paged decode attention.
 *
 * This file holds only random-number generation and the placement of generated
 * tokens into a paged pool. It contains none of the attention, quantisation or
 * merge arithmetic, so both the CPU oracle and the CUDA path can consume its
 * output without sharing any of the method's code.
 *
 * Generator (counter based, no hidden state):
 *   mix(z)      : the splitmix64 finaliser (Steele, Lea, Flood, "Fast splittable
 *                 pseudorandom number generators", OOPSLA 2014):
 *                 z ^= z >> 30; z *= 0xbf58476d1ce4e5b9;
 *                 z ^= z >> 27; z *= 0x94d049bb133111eb; z ^= z >> 31.
 *   key(s, t)   = mix(mix(s ^ 0x5851f42d4c957f2d) + t * GAMMA), GAMMA = 0x9e3779b97f4a7c15
 *   u64(s,t,i)  = mix(key(s, t) + (i + 1) * GAMMA)
 *   unif(s,t,i) = (u64 >> 11) * 2^-53                      in [0, 1)
 *   normal(s,t,i): Box-Muller on the pair (2i, 2i+1):
 *                 u1 = ((u64(2i) >> 11) + 1) * 2^-53        in (0, 1]
 *                 u2 = unif(2i + 1)
 *                 z  = sqrt(-2 ln u1) * cos(2 pi u2)        (double)
 *   bf16(x)     : x rounded to float (RNE), then to bfloat16 (RNE on the bits).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

#define GAMMA 0x9e3779b97f4a7c15ULL

static inline uint64_t mix64(uint64_t z) {
  z ^= z >> 30;
  z *= 0xbf58476d1ce4e5b9ULL;
  z ^= z >> 27;
  z *= 0x94d049bb133111ebULL;
  z ^= z >> 31;
  return z;
}

static inline uint64_t stream_key(uint64_t seed, uint64_t tid) {
  return mix64(mix64(seed ^ 0x5851f42d4c957f2dULL) + tid * GAMMA);
}

static inline uint64_t u64_at(uint64_t key, uint64_t i) { return mix64(key + (i + 1) * GAMMA); }

static inline double unif_at(uint64_t key, uint64_t i) {
  return (double)(u64_at(key, i) >> 11) * 0x1.0p-53;
}

static inline double normal_at(uint64_t key, uint64_t i) {
  double u1 = (double)((u64_at(key, 2 * i) >> 11) + 1) * 0x1.0p-53;
  double u2 = unif_at(key, 2 * i + 1);
  return sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925286766559 * u2);
}

static inline uint16_t to_bf16(double x) {
  float f = (float)x;
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7f800000u) == 0x7f800000u) return (uint16_t)((u >> 16) | ((u & 0xffffu) ? 0x40u : 0u));
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* ---------------------------------------------------------------- scalar API */

uint64_t tpks_u64(uint64_t seed, uint64_t tid, uint64_t i) { return u64_at(stream_key(seed, tid), i); }

void tpks_uniform(uint64_t seed, uint64_t tid, uint64_t offset, int64_t n, double* out) {
  uint64_t key = stream_key(seed, tid);
  for (int64_t i = 0; i < n; ++i) out[i] = unif_at(key, offset + (uint64_t)i);
}

void tpks_normal(uint64_t seed, uint64_t tid, uint64_t offset, int64_t n, double* out) {
  uint64_t key = stream_key(seed, tid);
  for (int64_t i = 0; i < n; ++i) out[i] = normal_at(key, offset + (uint64_t)i);
}

/* out[i] = bf16(normal(offset + i) * sigma[(offset + i) % period]); sigma may be NULL. */
void tpks_normal_bf16(uint64_t seed, uint64_t tid, uint64_t offset, int64_t n, const double* sigma,
                      int64_t period, uint16_t* out) {
  uint64_t key = stream_key(seed, tid);
  for (int64_t i = 0; i < n; ++i) {
    uint64_t g = offset + (uint64_t)i;
    double s = sigma ? sigma[g % (uint64_t)period] : 1.0;
    out[i] = to_bf16(normal_at(key, g) * s);
  }
}

/* Fisher-Yates shuffle of 0..n-1, swap index j = floor(unif(i) * (i + 1)) for i = n-1 .. 1. */
void tpks_permutation(uint64_t seed, uint64_t tid, int64_t n, int32_t* out) {
  uint64_t key = stream_key(seed, tid);
  for (int64_t i = 0; i < n; ++i) out[i] = (int32_t)i;
  for (int64_t i = n - 1; i > 0; --i) {
    int64_t j = (int64_t)(unif_at(key, (uint64_t)i) * (double)(i + 1));
    if (j > i) j = i;
    int32_t t = out[i];
    out[i] = out[j];
    out[j] = t;
  }
}

/* out[i] = lo + floor(unif(i) * (hi - lo + 1)), inclusive range. */
void tpks_randint(uint64_t seed, uint64_t tid, int64_t n, int64_t lo, int64_t hi, int64_t* out) {
  uint64_t key = stream_key(seed, tid);
  for (int64_t i = 0; i < n; ++i) {
    int64_t v = lo + (int64_t)(unif_at(key, (uint64_t)i) * (double)(hi - lo + 1));
    out[i] = v > hi ? hi : v;
  }
}

/* ------------------------------------------------------- paged pool filling */
/*
 * Fill the pages of one logical history into a paged pool laid out
 * [slot][heads][page_tokens][dim] (bfloat16).  Logical token `tok` of head `h`
 * takes the normals at index (h * n_tokens + tok) * dim + c, so the logical
 * history does not depend on which physical slot a page lands in.
 * sigma is [heads][dim] (or NULL for unit variance).  Tokens past n_tokens in
 * the last page are left untouched.
 */
typedef struct {
  uint64_t key;
  int heads, dim, page_tokens;
  int64_t n_tokens;
  const int32_t* slot_of_page;
  const double* sigma;
  uint16_t* pool;
  int64_t page_lo, page_hi;
} fill_job;

static void* fill_worker(void* arg) {
  fill_job* j = (fill_job*)arg;
  const int64_t page_elems = (int64_t)j->page_tokens * j->dim;
  for (int64_t p = j->page_lo; p < j->page_hi; ++p) {
    int64_t slot = j->slot_of_page[p];
    for (int h = 0; h < j->heads; ++h) {
      uint16_t* dst = j->pool + (slot * j->heads + h) * page_elems;
      for (int t = 0; t < j->page_tokens; ++t) {
        int64_t tok = p * j->page_tokens + t;
        if (tok >= j->n_tokens) break;
        uint64_t base = ((uint64_t)h * (uint64_t)j->n_tokens + (uint64_t)tok) * (uint64_t)j->dim;
        for (int c = 0; c < j->dim; ++c) {
          double s = j->sigma ? j->sigma[h * j->dim + c] : 1.0;
          dst[t * j->dim + c] = to_bf16(normal_at(j->key, base + (uint64_t)c) * s);
        }
      }
    }
  }
  return 0;
}

void tpks_fill_pages(uint64_t seed, uint64_t tid, int heads, int64_t n_tokens, int dim, int page_tokens,
                     const int32_t* slot_of_page, const double* sigma, uint16_t* pool, int n_threads) {
  int64_t n_pages = (n_tokens + page_tokens - 1) / page_tokens;
  if (n_threads < 1) n_threads = 1;
  if (n_threads > 256) n_threads = 256;
  if (n_pages < n_threads) n_threads = n_pages > 0 ? (int)n_pages : 1;
  pthread_t th[256];
  fill_job jobs[256];
  uint64_t key = stream_key(seed, tid);
  for (int i = 0; i < n_threads; ++i) {
    jobs[i].key = key;
    jobs[i].heads = heads;
    jobs[i].dim = dim;
    jobs[i].page_tokens = page_tokens;
    jobs[i].n_tokens = n_tokens;
    jobs[i].slot_of_page = slot_of_page;
    jobs[i].sigma = sigma;
    jobs[i].pool = pool;
    jobs[i].page_lo = n_pages * i / n_threads;
    jobs[i].page_hi = n_pages * (i + 1) / n_threads;
  }
  for (int i = 1; i < n_threads; ++i) pthread_create(&th[i], 0, fill_worker, &jobs[i]);
  fill_worker(&jobs[0]);
  for (int i = 1; i < n_threads; ++i) pthread_join(th[i], 0);
}
