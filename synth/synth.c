/*
 * synth.c — seeded synthetic inputs for block-sparse decode attention.
 *
 * This file is the one input generator that both the CUDA path's tests and
 * benchmark and the CPU oracle read from.  It holds none of the attention
 * method's arithmetic: it only turns (seed, stream, index) into numbers.
 *
 *   - Uniform 64-bit words come from SplitMix64 (Steele, Lea, Flood,
 *     "Fast splittable pseudorandom number generators", OOPSLA 2014) used as
 *     a counter-based generator: word i of a stream is mix(s0 + (i+1)*gamma),
 *     which is exactly the i-th output of a SplitMix64 generator seeded with
 *     s0.  Any element can therefore be produced on its own, in any order and
 *     on any number of threads, and always gets the same value.
 *   - Normal deviates use the Box-Muller transform (Box and Muller, 1958):
 *     element e uses the pair of words (2*(e/2), 2*(e/2)+1); even elements
 *     take the cosine branch, odd elements the sine branch.
 *   - Values are rounded once to IEEE 754 binary16 with round-to-nearest-even
 *     by an encoder written from the binary16 format definition.
 *
 * Build flags keep double arithmetic unfused (-ffp-contract=off) so that the
 * bytes do not depend on whether the compiler forms fused multiply-adds.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define SM64_GAMMA 0x9E3779B97F4A7C15ull

static inline uint64_t sm64_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

/* Start state of stream `stream` under `seed`. */
static inline uint64_t stream_base(uint64_t seed, uint64_t stream) {
  return sm64_mix(seed * SM64_GAMMA + sm64_mix(stream + SM64_GAMMA));
}

/* Word i of a stream: the (i+1)-th SplitMix64 output from the stream base. */
uint64_t synth_u64(uint64_t seed, uint64_t stream, uint64_t i) {
  return sm64_mix(stream_base(seed, stream) + (i + 1) * SM64_GAMMA);
}

void synth_fill_u64(uint64_t* out, uint64_t n, uint64_t seed, uint64_t stream,
                    uint64_t first) {
  uint64_t base = stream_base(seed, stream);
  for (uint64_t i = 0; i < n; ++i) out[i] = sm64_mix(base + (first + i + 1) * SM64_GAMMA);
}

/* Encode a double as binary16, round to nearest, ties to even. */
uint16_t synth_f16_from_double(double x) {
  uint16_t sign = signbit(x) ? 0x8000u : 0u;
  double a = fabs(x);
  if (isnan(x)) return 0x7E00u;
  if (a == 0.0) return sign;
  if (a >= 65520.0) return sign | 0x7C00u; /* halfway above 65504 ties to inf */
  int e2;
  (void)frexp(a, &e2);     /* a = f * 2^e2, f in [0.5, 1) */
  int E = e2 - 1;           /* a in [2^E, 2^(E+1)) */
  int qexp = (E < -14 ? -14 : E) - 10; /* binary16 quantum exponent */
  double m = ldexp(a, -qexp);           /* exact: power-of-two scaling */
  double r = rint(m);                   /* current mode: nearest-even */
  uint32_t mi = (uint32_t)r;
  if (qexp == -24) return (uint16_t)(sign | mi); /* subnormal (mi==1024 is 2^-14) */
  /* normal: value = mi * 2^qexp, mi in [1024, 2048]; mi==2048 carries. */
  uint32_t bits = ((uint32_t)(qexp + 25) << 10) + (mi - 1024u);
  return (uint16_t)(sign | bits);
}

/* Normal deviate for element e of a stream (Box-Muller). */
static inline double normal_at(uint64_t base, uint64_t e) {
  uint64_t p = e >> 1;
  uint64_t w0 = sm64_mix(base + (2 * p + 1) * SM64_GAMMA);
  uint64_t w1 = sm64_mix(base + (2 * p + 2) * SM64_GAMMA);
  double u1 = ((double)((w0 >> 11) + 1)) * 0x1.0p-53; /* (0, 1] */
  double u2 = ((double)(w1 >> 11)) * 0x1.0p-53;       /* [0, 1) */
  double r = sqrt(-2.0 * log(u1));
  double th = 6.283185307179586476925286766559 * u2;
  return (e & 1) ? r * sin(th) : r * cos(th);
}

typedef struct {
  uint16_t* out;
  uint64_t lo, hi, first, base;
  double mean, sigma;
  const double* chan_scale;
  int64_t d;
} fill_job;

static void* fill_worker(void* arg) {
  fill_job* j = (fill_job*)arg;
  for (uint64_t i = j->lo; i < j->hi; ++i) {
    uint64_t e = j->first + i;
    double s = j->sigma;
    if (j->chan_scale) s *= j->chan_scale[e % (uint64_t)j->d];
    j->out[i] = synth_f16_from_double(j->mean + s * normal_at(j->base, e));
  }
  return NULL;
}

/*
 * out[i] = f16(mean + sigma * chan_scale[(first+i) % d] * z(first+i)) for
 * i in [0, n).  chan_scale may be NULL (all ones).  nthreads <= 1 runs on the
 * calling thread; the bytes do not depend on nthreads.
 */
int synth_fill_normal_f16(uint16_t* out, uint64_t n, uint64_t seed, uint64_t stream,
                          uint64_t first, double mean, double sigma,
                          const double* chan_scale, int64_t d, int nthreads) {
  if (!out && n) return -1;
  if (chan_scale && d <= 0) return -1;
  uint64_t base = stream_base(seed, stream);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if ((uint64_t)nthreads > n / 65536 + 1) nthreads = (int)(n / 65536 + 1);
  fill_job jobs[256];
  pthread_t th[256];
  for (int t = 0; t < nthreads; ++t) {
    jobs[t].out = out;
    jobs[t].lo = n * (uint64_t)t / (uint64_t)nthreads;
    jobs[t].hi = n * (uint64_t)(t + 1) / (uint64_t)nthreads;
    jobs[t].first = first;
    jobs[t].base = base;
    jobs[t].mean = mean;
    jobs[t].sigma = sigma;
    jobs[t].chan_scale = chan_scale;
    jobs[t].d = d;
  }
  if (nthreads == 1) {
    fill_worker(&jobs[0]);
    return 0;
  }
  int started = 0;
  for (int t = 0; t < nthreads; ++t) {
    if (pthread_create(&th[t], NULL, fill_worker, &jobs[t]) != 0) break;
    ++started;
  }
  for (int t = started; t < nthreads; ++t) fill_worker(&jobs[t]); /* fallback */
  for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
  return 0;
}

/* Normal deviates as doubles (no rounding), for building derived inputs. */
void synth_fill_normal_f64(double* out, uint64_t n, uint64_t seed, uint64_t stream,
                           uint64_t first) {
  uint64_t base = stream_base(seed, stream);
  for (uint64_t i = 0; i < n; ++i) out[i] = normal_at(base, first + i);
}

void synth_f16_from_double_array(const double* in, uint16_t* out, uint64_t n) {
  for (uint64_t i = 0; i < n; ++i) out[i] = synth_f16_from_double(in[i]);
}
