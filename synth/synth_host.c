/*
 * Seeded synthetic inputs, host side.
 *
 * Counter-based: element `idx` of tensor `tid` under `seed` is drawn from the
 * (idx+1)-th output of SplitMix64 (Steele, Lea & Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014; the 64-bit finaliser
 * constants are Vigna's) seeded with key(seed, tid) = sm64((seed << 8) | tid).
 * Any slice of any tensor can therefore be regenerated without the rest.
 *
 *  - "normal" draws are an inverse-CDF table lookup: table[u >> 48], where the
 *    65536-entry table is built once in Python (synth/__init__.py) and passed
 *    in, so host and device read identical values;
 *  - "int" draws are uniform over {-a..a}: ((u >> 32) * (2a+1)) >> 32, minus a,
 *    optionally multiplied by a per-row integer factor (planted hot blocks).
 *
 * This file holds only input generation; it computes nothing of the method.
 * The device twin is synth_dev.cu; a GPU test checks the two agree bit for bit.
 */
#include <stdint.h>
#include <string.h>
#include <pthread.h>

#define SM64_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t sm64(uint64_t x) {
  uint64_t z = x + SM64_GAMMA;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

uint64_t synth_key(uint64_t seed, uint32_t tid) { return sm64((seed << 8) | (uint64_t)(tid & 0xFF)); }

uint64_t synth_u64(uint64_t key, uint64_t idx) { return sm64(key + idx * SM64_GAMMA); }

static inline uint16_t f32_to_bf16_bits_exact(float f) {
  /* values written here are already bf16-representable (table built that way,
     or small integers), so truncation is exact */
  uint32_t b;
  memcpy(&b, &f, 4);
  return (uint16_t)(b >> 16);
}

typedef struct {
  void* out;
  int out_kind; /* 0 = f32, 1 = bf16 bits */
  uint64_t n, start, key;
  const float* table; /* normal */
  int a;              /* int: range, <0 means normal */
  const uint8_t* row_mult;
  uint64_t row_len, rows_per_batch;
} job_t;

static void fill_range(const job_t* j, uint64_t lo, uint64_t hi) {
  for (uint64_t e = lo; e < hi; ++e) {
    uint64_t idx = j->start + e;
    uint64_t u = synth_u64(j->key, idx);
    float v;
    if (j->a < 0) {
      v = j->table[u >> 48];
    } else {
      uint64_t n = (uint64_t)(2 * j->a + 1);
      int64_t iv = (int64_t)(((u >> 32) * n) >> 32) - j->a;
      if (j->row_mult) {
        uint64_t row = (idx / j->row_len) % j->rows_per_batch;
        iv *= (int64_t)j->row_mult[row];
      }
      v = (float)iv;
    }
    if (j->out_kind == 0)
      ((float*)j->out)[e] = v;
    else
      ((uint16_t*)j->out)[e] = f32_to_bf16_bits_exact(v);
  }
}

typedef struct {
  const job_t* job;
  uint64_t lo, hi;
} part_t;

static void* worker(void* p) {
  const part_t* pt = (const part_t*)p;
  fill_range(pt->job, pt->lo, pt->hi);
  return 0;
}

static void run(const job_t* j, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (j->n < (1u << 16) || nthreads == 1) {
    fill_range(j, 0, j->n);
    return;
  }
  pthread_t th[256];
  part_t parts[256];
  uint64_t chunk = (j->n + nthreads - 1) / nthreads;
  int started = 0;
  for (int t = 0; t < nthreads; ++t) {
    parts[t].job = j;
    parts[t].lo = (uint64_t)t * chunk;
    parts[t].hi = parts[t].lo + chunk > j->n ? j->n : parts[t].lo + chunk;
    if (parts[t].lo >= parts[t].hi) break;
    if (pthread_create(&th[t], 0, worker, &parts[t]) != 0) {
      fill_range(j, parts[t].lo, parts[t].hi);
      parts[t].lo = parts[t].hi = 0;
      th[t] = 0;
    }
    started = t + 1;
  }
  for (int t = 0; t < started; ++t)
    if (parts[t].hi > parts[t].lo) pthread_join(th[t], 0);
}

/* out[e] = normal draw for flat index start+e, e in [0, n). */
void synth_fill_normal(void* out, int out_kind, uint64_t n, uint64_t start, uint64_t seed, uint32_t tid,
                       const float* table, int nthreads) {
  job_t j = {out, out_kind, n, start, synth_key(seed, tid), table, -1, 0, 1, 1};
  run(&j, nthreads);
}

/* out[e] = uniform integer in {-a..a} for flat index start+e, times
   row_mult[(idx / row_len) % rows_per_batch] when row_mult is given. */
void synth_fill_int(void* out, int out_kind, uint64_t n, uint64_t start, uint64_t seed, uint32_t tid, int a,
                    const uint8_t* row_mult, uint64_t row_len, uint64_t rows_per_batch, int nthreads) {
  job_t j = {out, out_kind, n, start, synth_key(seed, tid), 0, a, row_mult, row_len ? row_len : 1,
             rows_per_batch ? rows_per_batch : 1};
  run(&j, nthreads);
}
