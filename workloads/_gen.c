/* Counter-based SplitMix64 stream and Box-Muller normals, multi-threaded.
 * Same definition as workloads/__init__.py (the numpy statement of it):
 *   output k of seed s = mix(s + (k+1) * 0x9E3779B97F4A7C15)
 *   uniform = (output >> 11) * 2^-53
 *   normal pair p from outputs (2p, 2p+1): r = sqrt(-2 ln(1 - u1)), (r cos 2 pi u2, r sin 2 pi u2)
 * Holds no part of the attention arithmetic; it only draws inputs. */
#include <math.h>
#include <pthread.h>
#include <stdint.h>

static inline uint64_t sm64_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline double sm64_uniform(uint64_t seed, uint64_t k) {
  return (double)(sm64_mix(seed + (k + 1) * 0x9E3779B97F4A7C15ULL) >> 11) * 0x1.0p-53;
}

void sm64_fill(uint64_t seed, uint64_t start, uint64_t count, uint64_t* out) {
  for (uint64_t i = 0; i < count; ++i) out[i] = sm64_mix(seed + (start + i + 1) * 0x9E3779B97F4A7C15ULL);
}

typedef struct {
  uint64_t seed, start;  /* stream offset of the first output of pair 0 */
  int64_t n0, n1;        /* normals [n0, n1) of the request */
  float* out;
} job_t;

static void* normals_job(void* arg) {
  const job_t* j = (const job_t*)arg;
  const double two_pi = 6.283185307179586476925286766559;
  for (int64_t n = j->n0; n < j->n1; ++n) {
    const uint64_t pair = (uint64_t)n >> 1;
    const double u1 = sm64_uniform(j->seed, j->start + 2 * pair);
    const double u2 = sm64_uniform(j->seed, j->start + 2 * pair + 1);
    const double r = sqrt(-2.0 * log1p(-u1));
    const double t = two_pi * u2;
    j->out[n] = (float)((n & 1) ? r * sin(t) : r * cos(t));
  }
  return 0;
}

/* count normals rounded to fp32 (nearest even), from stream output `start`. */
void sm64_normals_f32(uint64_t seed, uint64_t start, int64_t count, float* out, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (count < (int64_t)1 << 16) nthreads = 1;
  pthread_t th[256];
  int created[256];
  job_t jobs[256];
  const int64_t per = ((count + nthreads - 1) / nthreads + 1) & ~(int64_t)1;
  for (int t = 0; t < nthreads; ++t) {
    created[t] = 0;
    int64_t a = per * t, b = a + per;
    if (a >= count) break;
    if (b > count) b = count;
    jobs[t].seed = seed;
    jobs[t].start = start;
    jobs[t].n0 = a;
    jobs[t].n1 = b;
    jobs[t].out = out;
    if (pthread_create(&th[t], 0, normals_job, &jobs[t]) == 0)
      created[t] = 1;
    else
      normals_job(&jobs[t]);
  }
  for (int t = 0; t < nthreads; ++t) {
    if (per * t >= count) break;
    if (created[t]) pthread_join(th[t], 0);
  }
}
