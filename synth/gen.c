/*
 * Seeded synthetic inputs for the MoE layer: a counter-based normal stream.
 *
 * This file holds no arithmetic of the MoE layer itself.  It draws numbers
 * and stores them in the formats the layer consumes (bf16, fp32, and a
 * block-scaled 4-bit encoding of weights).  Both the fp64 oracle and the
 * GPU path read the same arrays produced here; neither one's code lives here.
 *
 * Stream definition (fixed; every value is a pure function of its index):
 *   mix(z)          = the splitmix64 output finaliser
 *                     z ^= z>>30; z *= 0xBF58476D1CE4E5B9;
 *                     z ^= z>>27; z *= 0x94D049BB133111EB; z ^= z>>31
 *   key(seed, id)   = mix(seed ^ mix((id + 1) * 0x9E3779B97F4A7C15))
 *   bits(key, c)    = mix(key + (c + 1) * 0x9E3779B97F4A7C15)
 *   element i of stream (seed, id), pair p = i >> 1:
 *     u1 = ((bits(key, 2p)   >> 11) + 1) * 2^-53      in (0, 1]
 *     u2 =  (bits(key, 2p+1) >> 11)      * 2^-53      in [0, 1)
 *     r  = sqrt(-2 ln u1),  th = 2 pi u2               (Box-Muller)
 *     z_i = r cos th  (i even),  r sin th  (i odd)
 * Scaled normals are mean + std * z_i computed in double.
 *
 * bf16 storage rounds the double to float (round-to-nearest-even, the C
 * conversion) and then the float to bf16 (round-to-nearest-even on bits).
 *
 * The 4-bit weight encoding (32-element blocks, e2m1 codes, e8m0 scale byte)
 * follows the OCP Microscaling Formats v1.0 specification: the block's shared
 * exponent is floor(log2(max|w|)) - 2 (2 = the largest e2m1 exponent), every
 * element is divided by 2^exp and rounded to the nearest e2m1 magnitude
 * {0, .5, 1, 1.5, 2, 3, 4, 6} with ties to the even code and saturation at 6.
 * Byte j of a block holds element 2j in its low nibble and 2j+1 in its high
 * nibble; bit 3 of a nibble is the sign.
 *
 * Compiled with -ffp-contract=off so that x86-64 and aarch64 builds evaluate
 * the same expression trees (libm may still differ in the last bit across
 * machines; inputs are always generated on the host that uses them).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z ^= z >> 30;
  z *= 0xBF58476D1CE4E5B9ULL;
  z ^= z >> 27;
  z *= 0x94D049BB133111EBULL;
  z ^= z >> 31;
  return z;
}

static inline uint64_t stream_key(uint64_t seed, uint32_t id) {
  return mix64(seed ^ mix64(((uint64_t)id + 1ULL) * GOLDEN));
}

static inline uint64_t stream_bits(uint64_t key, uint64_t c) {
  return mix64(key + (c + 1ULL) * GOLDEN);
}

static inline double std_normal(uint64_t key, uint64_t i) {
  const uint64_t p = i >> 1;
  const double u1 = (double)((stream_bits(key, 2 * p) >> 11) + 1ULL) * 0x1.0p-53;
  const double u2 = (double)(stream_bits(key, 2 * p + 1) >> 11) * 0x1.0p-53;
  const double r = sqrt(-2.0 * log(u1));
  const double th = 6.283185307179586476925286766559 * u2;
  return (i & 1ULL) ? r * sin(th) : r * cos(th);
}

static inline uint16_t f64_to_bf16_bits(double v) {
  float f = (float)v;
  uint32_t b;
  memcpy(&b, &f, 4);
  if ((b & 0x7F800000u) == 0x7F800000u && (b & 0x007FFFFFu)) return 0x7FC0;
  b += 0x7FFFu + ((b >> 16) & 1u);
  return (uint16_t)(b >> 16);
}

/* ---- threading helper: split [0, n) into contiguous ranges ---- */
typedef struct {
  int kind;
  uint64_t key;
  uint64_t start, lo, hi;
  double mean, std;
  void* out;
  void* out2;
} job_t;

enum { K_F64 = 0, K_F32 = 1, K_BF16 = 2, K_MXFP4 = 3 };

static uint8_t e2m1_encode(double q) {
  /* q already divided by the block scale; returns a 4-bit code */
  const double a = fabs(q);
  uint8_t m;
  if (a <= 0.25) m = 0;          /* tie at .25 -> code 0 (even) */
  else if (a < 0.75) m = 1;
  else if (a <= 1.25) m = 2;     /* ties .75 and 1.25 -> code 2 (even) */
  else if (a < 1.75) m = 3;
  else if (a <= 2.5) m = 4;      /* ties 1.75 and 2.5 -> code 4 (even) */
  else if (a < 3.5) m = 5;
  else if (a <= 5.0) m = 6;      /* ties 3.5 and 5 -> code 6 (even) */
  else m = 7;                    /* (5, inf) -> 6.0, saturating */
  if (m != 0 && q < 0) m |= 8;
  return m;
}

static void run_range(job_t* j) {
  for (uint64_t n = j->lo; n < j->hi; ++n) {
    if (j->kind == K_MXFP4) {
      /* n is a block index; elements 32*(start+n) .. +32 of the stream */
      const uint64_t b = j->start + n;
      double w[32];
      double amax = 0.0;
      for (int i = 0; i < 32; ++i) {
        w[i] = j->mean + j->std * std_normal(j->key, 32 * b + (uint64_t)i);
        if (fabs(w[i]) > amax) amax = fabs(w[i]);
      }
      int e;
      if (amax == 0.0) {
        e = -127;
      } else {
        int ex;
        frexp(amax, &ex); /* amax = m * 2^ex, m in [0.5, 1) */
        e = (ex - 1) - 2;
        if (e < -127) e = -127;
        if (e > 127) e = 127;
      }
      ((uint8_t*)j->out2)[n] = (uint8_t)(e + 127);
      uint8_t* codes = (uint8_t*)j->out + 16 * n;
      for (int i = 0; i < 16; ++i) {
        const uint8_t lo = e2m1_encode(ldexp(w[2 * i], -e));
        const uint8_t hi = e2m1_encode(ldexp(w[2 * i + 1], -e));
        codes[i] = (uint8_t)(lo | (hi << 4));
      }
      continue;
    }
    const double v = j->mean + j->std * std_normal(j->key, j->start + n);
    switch (j->kind) {
      case K_F64: ((double*)j->out)[n] = v; break;
      case K_F32: ((float*)j->out)[n] = (float)v; break;
      default: ((uint16_t*)j->out)[n] = f64_to_bf16_bits(v); break;
    }
  }
}

static void* thread_main(void* arg) {
  run_range((job_t*)arg);
  return NULL;
}

static int g_threads = 0;

void synth_set_threads(int n) { g_threads = n; }

static void run_parallel(job_t base, uint64_t n) {
  int nt = g_threads > 0 ? g_threads : 8;
  if (n < 65536 || nt <= 1) {
    base.lo = 0;
    base.hi = n;
    run_range(&base);
    return;
  }
  if (nt > 64) nt = 64;
  pthread_t th[64];
  job_t jobs[64];
  int started[64] = {0};
  for (int t = 0; t < nt; ++t) {
    jobs[t] = base;
    jobs[t].lo = n * (uint64_t)t / (uint64_t)nt;
    jobs[t].hi = n * (uint64_t)(t + 1) / (uint64_t)nt;
    started[t] = pthread_create(&th[t], NULL, thread_main, &jobs[t]) == 0;
    if (!started[t]) run_range(&jobs[t]);
  }
  for (int t = 0; t < nt; ++t)
    if (started[t]) pthread_join(th[t], NULL);
}

static job_t make_job(int kind, uint64_t seed, uint32_t id, uint64_t start, double mean, double std,
                      void* out, void* out2) {
  job_t j;
  memset(&j, 0, sizeof j);
  j.kind = kind;
  j.key = stream_key(seed, id);
  j.start = start;
  j.mean = mean;
  j.std = std;
  j.out = out;
  j.out2 = out2;
  return j;
}

/* Elements [start, start+count) of stream (seed, id), as mean + std * z. */
void synth_normal_f64(uint64_t seed, uint32_t id, uint64_t start, uint64_t count, double mean,
                      double std, double* out) {
  run_parallel(make_job(K_F64, seed, id, start, mean, std, out, NULL), count);
}

void synth_normal_f32(uint64_t seed, uint32_t id, uint64_t start, uint64_t count, double mean,
                      double std, float* out) {
  run_parallel(make_job(K_F32, seed, id, start, mean, std, out, NULL), count);
}

void synth_normal_bf16(uint64_t seed, uint32_t id, uint64_t start, uint64_t count, double mean,
                       double std, uint16_t* out) {
  run_parallel(make_job(K_BF16, seed, id, start, mean, std, out, NULL), count);
}

/* Blocks [start_block, start_block+nblocks) of 32 elements each: 16 code bytes
 * per block into codes, one e8m0 byte per block into scales. */
void synth_mxfp4(uint64_t seed, uint32_t id, uint64_t start_block, uint64_t nblocks, double std,
                 uint8_t* codes, uint8_t* scales) {
  run_parallel(make_job(K_MXFP4, seed, id, start_block, 0.0, std, codes, scales), nblocks);
}

/* Round doubles to bf16 bits (double -> float -> bf16, both nearest-even). */
void synth_round_bf16(const double* in, uint64_t n, uint16_t* out) {
  for (uint64_t i = 0; i < n; ++i) out[i] = f64_to_bf16_bits(in[i]);
}
