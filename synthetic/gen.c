/* Counter-based normal generator for the synthetic inputs of the Ulysses block.
 *
 * Test and benchmark infrastructure: it draws the seeded inputs (X, W_qkv, dO, Q/K/V)
 * that both the CPU oracle and the GPU library are fed.  It holds none of the
 * attention block's arithmetic.
 *
 * Definition (one value per index n of a tensor identified by (seed, tensor_id)):
 *   key      = mix64(seed * 2^32 + tensor_id)
 *   x(c)     = mix64(key + c * 0x9E3779B97F4A7C15),  c = 1, 2, ...   (SplitMix64 stream)
 *   u1       = ((x(2n+1) >> 11) + 1) * 2^-53                        in (0, 1]
 *   u2       =  (x(2n+2) >> 11)      * 2^-53                        in [0, 1)
 *   z        = sqrt(-2 ln u1) * cos(2 pi u2)                        (Box-Muller, cosine branch)
 *   value    = bf16_rne(float32_rne(mean + std * z))
 * mix64 is the SplitMix64 finaliser of Steele, Lea and Flood (OOPSLA 2014):
 *   z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9; z = (z ^ (z >> 27)) * 0x94D049BB133111EB;
 *   z ^ (z >> 31).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  uint32_t bias = 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)((u + bias) >> 16);
}

typedef struct {
  uint64_t key, begin, end;
  double mean, std;
  uint16_t *out_bf16;
  double *out_f64;
} job_t;

static const double kTwoPi = 6.283185307179586476925286766559;
static const double kTwoPowM53 = 1.1102230246251565404236316680908203125e-16;
static const uint64_t kGamma = 0x9E3779B97F4A7C15ULL;

static void *run_job(void *arg) {
  job_t *j = (job_t *)arg;
  for (uint64_t n = j->begin; n < j->end; ++n) {
    uint64_t a = mix64(j->key + (2 * n + 1) * kGamma);
    uint64_t b = mix64(j->key + (2 * n + 2) * kGamma);
    double u1 = (double)((a >> 11) + 1) * kTwoPowM53;
    double u2 = (double)(b >> 11) * kTwoPowM53;
    double z = sqrt(-2.0 * log(u1)) * cos(kTwoPi * u2);
    double v = j->mean + j->std * z;
    if (j->out_bf16) j->out_bf16[n - j->begin] = f32_to_bf16_rne((float)v);
    if (j->out_f64) j->out_f64[n - j->begin] = v;
  }
  return 0;
}

/* Writes values [offset, offset+count) of tensor (seed, tensor_id).  Either output may be
 * NULL.  nthreads <= 1 runs on the calling thread.  Returns 0. */
int synth_normal(uint64_t seed, uint64_t tensor_id, uint64_t offset, uint64_t count,
                 double mean, double std, uint16_t *out_bf16, double *out_f64,
                 int nthreads) {
  uint64_t key = mix64(seed * 4294967296ULL + tensor_id);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if ((uint64_t)nthreads > count / 65536 + 1) nthreads = (int)(count / 65536 + 1);
  job_t jobs[256];
  pthread_t th[256];
  int created[256];
  uint64_t per = (count + nthreads - 1) / nthreads;
  for (int t = 0; t < nthreads; ++t) {
    uint64_t b = offset + per * t, e = b + per;
    if (e > offset + count) e = offset + count;
    if (b > e) b = e;
    jobs[t].key = key;
    jobs[t].begin = b;
    jobs[t].end = e;
    jobs[t].mean = mean;
    jobs[t].std = std;
    jobs[t].out_bf16 = out_bf16 ? out_bf16 + (b - offset) : 0;
    jobs[t].out_f64 = out_f64 ? out_f64 + (b - offset) : 0;
    created[t] = 0;
    if (t == 0 || b == e) continue;
    created[t] = pthread_create(&th[t], 0, run_job, &jobs[t]) == 0;
    if (!created[t]) run_job(&jobs[t]);
  }
  run_job(&jobs[0]);
  for (int t = 1; t < nthreads; ++t)
    if (created[t]) pthread_join(th[t], 0);
  return 0;
}
