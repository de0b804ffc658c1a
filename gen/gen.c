/*
 * Seeded, counter-based generator of synthetic attention inputs.
 *
 * It holds none of the attention method's arithmetic: it only turns
 * (seed, tensor id, flat index) into bits, uniforms, normals and bf16 codes.
 * Both the CUDA path and the CPU oracle consume the bytes it writes.
 *
 * Counter-based PRNG: SplitMix64 (Steele, Lea and Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014), used in its stateless form
 * r(i) = mix(key + (i + 1) * gamma) with gamma the 64-bit golden ratio.
 * Normals: Box-Muller (1958) on pairs of uniforms. bf16: the upper 16 bits of
 * an IEEE float32 after round-to-nearest-even.
 *
 * Portable C99 + pthreads; no architecture-specific code.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

#define GEN_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t gen_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

/* Key of one stream: one per (seed, tensor id). */
static inline uint64_t gen_key(uint64_t seed, uint32_t tensor_id) {
  uint64_t a = gen_mix(seed + GEN_GAMMA);
  return gen_mix(a + (uint64_t)(tensor_id + 1) * GEN_GAMMA);
}

static inline uint64_t gen_bits(uint64_t key, uint64_t i) {
  return gen_mix(key + (i + 1) * GEN_GAMMA);
}

/* Uniform in [0, 1): top 53 bits. */
static inline double gen_u01(uint64_t r) { return (double)(r >> 11) * (1.0 / 9007199254740992.0); }
/* Uniform in (0, 1]: never 0, so log() below stays finite. */
static inline double gen_u01_open0(uint64_t r) { return (double)((r >> 11) + 1) * (1.0 / 9007199254740992.0); }

static inline uint16_t gen_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)0x7FC0; /* NaN */
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

/* Standard normal for flat index i: element 2p uses the cosine branch and
 * element 2p+1 the sine branch of the same Box-Muller pair p. */
static inline double gen_normal_at(uint64_t key, uint64_t i) {
  uint64_t p = i >> 1;
  double u1 = gen_u01_open0(gen_bits(key, 2 * p));
  double u2 = gen_u01(gen_bits(key, 2 * p + 1));
  double rad = sqrt(-2.0 * log(u1));
  double ang = 6.283185307179586 * u2;
  return (i & 1) ? rad * sin(ang) : rad * cos(ang);
}

typedef struct {
  uint16_t* out;
  int64_t begin, end;
  uint64_t key;
  double a, b;
  int kind; /* 0 normal(mu=a, sigma=b), 1 uniform[a, b) */
} gen_job;

static void* gen_worker(void* arg) {
  gen_job* j = (gen_job*)arg;
  for (int64_t i = j->begin; i < j->end; ++i) {
    double x;
    if (j->kind == 0)
      x = j->a + j->b * gen_normal_at(j->key, (uint64_t)i);
    else
      x = j->a + (j->b - j->a) * gen_u01(gen_bits(j->key, (uint64_t)i));
    j->out[i] = gen_f32_to_bf16((float)x);
  }
  return NULL;
}

#define GEN_MAX_THREADS 64

static int gen_fill(uint16_t* out, int64_t n, uint64_t seed, uint32_t tensor_id, double a, double b,
                    int kind, int threads) {
  if (n < 0 || (n > 0 && !out)) return -1;
  if (threads < 1) threads = 1;
  if (threads > GEN_MAX_THREADS) threads = GEN_MAX_THREADS;
  if (n < (int64_t)1 << 16) threads = 1;
  gen_job jobs[GEN_MAX_THREADS];
  pthread_t tids[GEN_MAX_THREADS];
  uint64_t key = gen_key(seed, tensor_id);
  int64_t per = (n + threads - 1) / threads;
  for (int t = 0; t < threads; ++t) {
    int64_t b0 = (int64_t)t * per, b1 = b0 + per < n ? b0 + per : n;
    jobs[t] = (gen_job){out, b0, b1 > b0 ? b1 : b0, key, a, b, kind};
    if (t == 0) continue;
    if (pthread_create(&tids[t], NULL, gen_worker, &jobs[t]) != 0) {
      gen_worker(&jobs[t]); /* run inline if a thread cannot start */
      tids[t] = 0;
    }
  }
  gen_worker(&jobs[0]);
  for (int t = 1; t < threads; ++t)
    if (tids[t]) pthread_join(tids[t], NULL);
  return 0;
}

/* n bf16 codes of N(mu, sigma^2). */
int gen_normal_bf16(uint16_t* out, int64_t n, uint64_t seed, uint32_t tensor_id, double mu, double sigma,
                    int threads) {
  return gen_fill(out, n, seed, tensor_id, mu, sigma, 0, threads);
}

/* n bf16 codes of U[lo, hi). */
int gen_uniform_bf16(uint16_t* out, int64_t n, uint64_t seed, uint32_t tensor_id, double lo, double hi,
                     int threads) {
  return gen_fill(out, n, seed, tensor_id, lo, hi, 1, threads);
}

/* n integers uniform on [lo, hi] (inclusive), by multiply-shift of a 53-bit uniform. */
int gen_uniform_int(int32_t* out, int64_t n, uint64_t seed, uint32_t tensor_id, int32_t lo, int32_t hi) {
  if (n < 0 || (n > 0 && !out) || hi < lo) return -1;
  uint64_t key = gen_key(seed, tensor_id);
  double span = (double)hi - (double)lo + 1.0;
  for (int64_t i = 0; i < n; ++i) {
    int64_t v = (int64_t)lo + (int64_t)floor(gen_u01(gen_bits(key, (uint64_t)i)) * span);
    if (v > hi) v = hi;
    out[i] = (int32_t)v;
  }
  return 0;
}

/* Raw 64-bit stream words, for tests of the stream itself. */
int gen_raw_u64(uint64_t* out, int64_t n, uint64_t seed, uint32_t tensor_id) {
  if (n < 0 || (n > 0 && !out)) return -1;
  uint64_t key = gen_key(seed, tensor_id);
  for (int64_t i = 0; i < n; ++i) out[i] = gen_bits(key, (uint64_t)i);
  return 0;
}

/* SplitMix64 sequence from a seed in its usual stateful form (state += gamma;
 * return mix(state)), exposed so a test can check the mixer against the
 * published first outputs. */
int gen_splitmix64_sequence(uint64_t* out, int64_t n, uint64_t seed) {
  if (n < 0 || (n > 0 && !out)) return -1;
  uint64_t s = seed;
  for (int64_t i = 0; i < n; ++i) {
    s += GEN_GAMMA;
    out[i] = gen_mix(s);
  }
  return 0;
}
