/* Online-softmax attention forward on the host CPU (include/attn_cpu.h).
 *
 * Work: units of (batch, head, 64-row query tile), handed out by an atomic counter to
 * the worker threads (causal tiles longest first).  A unit keeps its query tile
 * (converted to fp32), the running max m, denominator l and accumulator o~ of its rows
 * in a per-thread buffer, and streams the visible key blocks of 64 rows through it:
 *
 *   for each key block:  s = q . k for the block (dot products over d, vectorised),
 *                        masked keys -inf before the max, m_new = max(m, max s),
 *                        alpha = exp(m - m_new), p = exp(s - m_new),
 *                        l = alpha l + sum p,  o~ = alpha o~ + sum p v
 *   at the end:          O = o~ / l (bf16), LSE = m + ln l; l = 0 gives O = 0, LSE = -inf
 *
 * ("FlashAttention math", sections "The block-wise update, and the full algorithm" and
 * "Pitfalls in implementing the recurrence"; while a row has seen no visible key its
 * reference is 0, so alpha = p = 0.)  The inner loops run over contiguous fp32 rows of
 * length d and are written for the compiler to vectorise (OpenMP simd pragmas; no
 * intrinsics, so the same source builds on x86-64 and aarch64).
 */
#include "../../include/attn_cpu.h"

#include <math.h>
#include <pthread.h>
#include <stdatomic.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define BQ 64 /* query rows per tile */
#define BK 64 /* keys per block */
#define DMAX 256

static float bf16_to_f32(uint16_t c) {
  uint32_t u = (uint32_t)c << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* round to nearest even; the values here are finite */
static uint16_t f32_to_bf16(float x) {
  uint32_t u;
  memcpy(&u, &x, sizeof u);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* keys j < limit(row) are visible: padding and the bottom-right causal bound */
static int row_limit(int row, int kv_len, int Nq, int Nk, int causal) {
  if (!causal) return kv_len;
  long long lim = (long long)row + Nk - Nq + 1;
  if (lim < 0) lim = 0;
  return lim < kv_len ? (int)lim : kv_len;
}

typedef struct {
  const uint16_t *Q, *K, *V;
  uint16_t* O;
  float* LSE;
  int B, H, Nq, Nk, d, causal, nqt;
  float scale;
  const int32_t* lens;
  long long units;
  atomic_llong next;
} job_t;

typedef struct {
  float q[BQ * DMAX];
  float k[BK * DMAX];
  float v[BK * DMAX];
  float o[BQ * DMAX];
  float s[BK];
  float m[BQ], l[BQ];
} scratch_t;

static void run_unit(const job_t* jb, long long u, scratch_t* w) {
  const int d = jb->d, nqt = jb->nqt;
  const long long bh = u / nqt;
  int qt = (int)(u % nqt);
  if (jb->causal) qt = nqt - 1 - qt; /* longest tiles first */
  const int b = (int)(bh / jb->H);
  const int q0 = qt * BQ;
  const int q1 = q0 + BQ < jb->Nq ? q0 + BQ : jb->Nq;
  const int rows = q1 - q0;
  int kv_len = jb->Nk;
  if (jb->lens) {
    const int L = jb->lens[b];
    kv_len = L < 0 ? 0 : (L > jb->Nk ? jb->Nk : L);
  }
  const uint16_t* Qh = jb->Q + ((size_t)bh * jb->Nq + q0) * d;
  const uint16_t* Kh = jb->K ? jb->K + (size_t)bh * jb->Nk * d : NULL;
  const uint16_t* Vh = jb->V ? jb->V + (size_t)bh * jb->Nk * d : NULL;
  for (int i = 0; i < rows; ++i) {
    for (int x = 0; x < d; ++x) w->q[i * d + x] = bf16_to_f32(Qh[(size_t)i * d + x]) * jb->scale;
    for (int x = 0; x < d; ++x) w->o[i * d + x] = 0.f;
    w->m[i] = -INFINITY;
    w->l[i] = 0.f;
  }
  const int kend = row_limit(q1 - 1, kv_len, jb->Nq, jb->Nk, jb->causal); /* the widest row */
  for (int k0 = 0; k0 < kend; k0 += BK) {
    const int kn = k0 + BK < kend ? BK : kend - k0;
    for (int j = 0; j < kn; ++j)
      for (int x = 0; x < d; ++x) {
        w->k[j * d + x] = bf16_to_f32(Kh[(size_t)(k0 + j) * d + x]);
        w->v[j * d + x] = bf16_to_f32(Vh[(size_t)(k0 + j) * d + x]);
      }
    for (int i = 0; i < rows; ++i) {
      const int lim = row_limit(q0 + i, kv_len, jb->Nq, jb->Nk, jb->causal);
      const int jn = lim - k0 < kn ? lim - k0 : kn; /* visible keys of this block */
      if (jn <= 0) continue;                        /* masked: contributes nothing */
      const float* qi = w->q + i * d;
      float mb = -INFINITY;
      for (int j = 0; j < jn; ++j) {
        const float* kj = w->k + j * d;
        float acc = 0.f;
#pragma omp simd reduction(+ : acc)
        for (int x = 0; x < d; ++x) acc += qi[x] * kj[x];
        w->s[j] = acc;
        mb = acc > mb ? acc : mb;
      }
      const float m_old = w->m[i];
      const float m_new = mb > m_old ? mb : m_old;
      const float alpha = expf(m_old - m_new); /* 0 when m_old = -inf */
      float lsum = 0.f;
      for (int j = 0; j < jn; ++j) {
        w->s[j] = expf(w->s[j] - m_new);
        lsum += w->s[j];
      }
      w->l[i] = alpha * w->l[i] + lsum;
      w->m[i] = m_new;
      float* oi = w->o + i * d;
      if (alpha != 1.f) {
#pragma omp simd
        for (int x = 0; x < d; ++x) oi[x] *= alpha;
      }
      for (int j = 0; j < jn; ++j) {
        const float pj = w->s[j];
        const float* vj = w->v + j * d;
#pragma omp simd
        for (int x = 0; x < d; ++x) oi[x] += pj * vj[x];
      }
    }
  }
  uint16_t* Oh = jb->O + ((size_t)bh * jb->Nq + q0) * d;
  float* Lh = jb->LSE + (size_t)bh * jb->Nq + q0;
  for (int i = 0; i < rows; ++i) {
    const float l = w->l[i];
    const float inv = l > 0.f ? 1.f / l : 0.f;
    for (int x = 0; x < d; ++x) Oh[(size_t)i * d + x] = f32_to_bf16(w->o[i * d + x] * inv);
    Lh[i] = l > 0.f ? w->m[i] + logf(l) : -INFINITY;
  }
}

static void* worker(void* arg) {
  job_t* jb = (job_t*)arg;
  scratch_t* w = (scratch_t*)malloc(sizeof(scratch_t));
  if (!w) return (void*)1;
  for (;;) {
    const long long u = atomic_fetch_add(&jb->next, 1);
    if (u >= jb->units) break;
    run_unit(jb, u, w);
  }
  free(w);
  return NULL;
}

attn_status attn_fwd_cpu(const uint16_t* Q, const uint16_t* K, const uint16_t* V, uint16_t* O, float* LSE, int B,
                         int H, int Nq, int Nk, int d, float scale, int causal, const int32_t* key_padding_lens,
                         int num_threads) {
  if (B < 0 || H < 0 || Nq < 0 || Nk < 0) return ATTN_ERR_BAD_SHAPE;
  if (d < 1 || d > DMAX) return ATTN_ERR_UNSUPPORTED_D;
  if (!(scale > 0.f) || !isfinite(scale) || num_threads < 0) return ATTN_ERR_BAD_ARG;
  if ((long long)B * H == 0 || Nq == 0) return ATTN_OK;
  if (!Q || !O || !LSE || (Nk > 0 && (!K || !V))) return ATTN_ERR_NULLPTR;
  job_t jb;
  jb.Q = Q;
  jb.K = Nk > 0 ? K : NULL;
  jb.V = Nk > 0 ? V : NULL;
  jb.O = O;
  jb.LSE = LSE;
  jb.B = B;
  jb.H = H;
  jb.Nq = Nq;
  jb.Nk = Nk;
  jb.d = d;
  jb.causal = causal ? 1 : 0;
  jb.scale = scale;
  jb.lens = key_padding_lens;
  jb.nqt = (Nq + BQ - 1) / BQ;
  jb.units = (long long)B * H * jb.nqt;
  atomic_init(&jb.next, 0);
  long n = num_threads > 0 ? num_threads : sysconf(_SC_NPROCESSORS_ONLN);
  if (n < 1) n = 1;
  if (n > jb.units) n = (long)jb.units;
  pthread_t* th = (pthread_t*)calloc((size_t)n, sizeof(pthread_t));
  int started = 0;
  attn_status st = ATTN_OK;
  if (th) {
    for (long t = 1; t < n; ++t) {
      if (pthread_create(&th[t], NULL, worker, &jb) != 0) {
        st = ATTN_ERR_LAUNCH;
        break;
      }
      ++started;
    }
  }
  if (worker(&jb) != NULL) st = ATTN_ERR_LAUNCH; /* the calling thread works too */
  for (int t = 1; t <= started; ++t) {
    void* r = NULL;
    pthread_join(th[t], &r);
    if (r != NULL) st = ATTN_ERR_LAUNCH;
  }
  free(th);
  return st;
}
