/*
 * Seeded synthetic workload generator for the MSA decode path.
 *
 * Produces the INPUTS of the path: FP8 E4M3 queries and NVFP4 paged caches
 * (E2M1 codes + one E4M3 scale per 16 elements, scale = E4M3(amax / 6)),
 * from N(0,1) values drawn by a counter-based generator, so every value is a
 * pure function of (seed, stream, index) and the output does not depend on the
 * number of threads or on the machine. None of the path's arithmetic (the
 * dequantisation, scores, pooling, selection or attention) lives here.
 *
 * Normal variates: splitmix64 over (seed, stream, pair index) gives two
 * uniforms; the Box-Muller transform turns them into two N(0,1) values, the
 * cosine branch for even indices and the sine branch for odd ones.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static inline uint64_t splitmix64(uint64_t z) {
  z += 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

static inline uint64_t key_of(uint64_t seed, uint64_t stream) {
  return splitmix64(splitmix64(seed * 0x2545F4914F6CDD1Dull + 0x1234567ull) ^ (stream * 0x9E3779B97F4A7C15ull));
}

/* uniform in (0, 1]: 53 random bits */
static inline double unit_open0(uint64_t x) { return ((double)(x >> 11) + 1.0) * (1.0 / 9007199254740992.0); }
static inline double unit_closed0(uint64_t x) { return (double)(x >> 11) * (1.0 / 9007199254740992.0); }

/* The pair (2p, 2p+1) of stream key k: cosine and sine branches. */
static inline void normal_pair(uint64_t k, uint64_t p, double* c, double* s) {
  double u1 = unit_open0(splitmix64(k ^ (2 * p))), u2 = unit_closed0(splitmix64(k ^ (2 * p + 1)));
  double r = sqrt(-2.0 * log(u1)), th = 6.283185307179586 * u2;
  *c = r * cos(th);
  *s = r * sin(th);
}

double synth_normal(uint64_t seed, uint64_t stream, uint64_t i) {
  double c, s;
  normal_pair(key_of(seed, stream), i >> 1, &c, &s);
  return (i & 1) ? s : c;
}

uint64_t synth_u64(uint64_t seed, uint64_t stream, uint64_t i) {
  return splitmix64(key_of(seed, stream) ^ (i * 0xD1B54A32D192ED03ull + 0x5BD1E995ull));
}

/* ---- encoders used to produce the inputs ---- */

/* E4M3 (OCP FN) encode: nearest, ties to even, saturate to +-448, NaN -> 0x7F.
 * Bit-level: exponent from frexp, mantissa rounded with rint (ties to even). */
static uint8_t enc_e4m3(double x) {
  uint8_t sign = signbit(x) ? 0x80 : 0;
  double a = fabs(x);
  int e;
  double m;
  if (isnan(x)) return 0x7F;
  if (a >= 448.0) return sign | 0x7E;
  if (a < ldexp(1.0, -6)) {                 /* subnormal grid: multiples of 2^-9 */
    double q = rint(a * 512.0);             /* 0..8; 8 == smallest normal, code 0x08 */
    return sign | (uint8_t)q;
  }
  m = frexp(a, &e);                         /* a = m * 2^e, m in [0.5, 1) */
  {
    double frac = rint((2.0 * m - 1.0) * 8.0);  /* 3 mantissa bits, 0..8 */
    int ex = e - 1 + 7;
    if (frac >= 8.0) { frac = 0.0; ex += 1; }
    if (ex > 15 || (ex == 15 && frac >= 7.0)) return sign | 0x7E;
    return sign | (uint8_t)((ex << 3) | (int)frac);
  }
}

static double dec_e4m3(uint8_t b) {
  int s = b >> 7, e = (b >> 3) & 15, m = b & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  v = e ? ldexp(1.0 + m / 8.0, e - 7) : ldexp((double)m, -9);
  return s ? -v : v;
}

/* E2M1 encode of a value already divided by its scale: nearest of
 * {0, .5, 1, 1.5, 2, 3, 4, 6}, ties to the even code, saturate at 6. */
static uint8_t enc_e2m1(double x) {
  uint8_t sign = signbit(x) ? 8 : 0;
  double a = fabs(x);
  uint8_t c;
  if (a <= 0.25) c = 0;
  else if (a < 0.75) c = 1;
  else if (a <= 1.25) c = 2;
  else if (a < 1.75) c = 3;
  else if (a <= 2.5) c = 4;
  else if (a < 3.5) c = 5;
  else if (a <= 5.0) c = 6;
  else c = 7;
  return sign | c;
}

/* NVFP4-encode one 128-element row: 8 groups of 16, scale = E4M3(amax/6). */
static void enc_nvfp4_row(const double* x, uint8_t* codes, uint8_t* scales) {
  int g, j;
  for (g = 0; g < 8; g++) {
    double amax = 0.0, sv;
    for (j = 0; j < 16; j++) { double a = fabs(x[g * 16 + j]); if (a > amax) amax = a; }
    scales[g] = enc_e4m3(amax / 6.0);
    sv = dec_e4m3(scales[g]);
    for (j = 0; j < 16; j += 2) {
      uint8_t lo = sv > 0 ? enc_e2m1(x[g * 16 + j] / sv) : 0;
      uint8_t hi = sv > 0 ? enc_e2m1(x[g * 16 + j + 1] / sv) : 0;
      codes[(g * 16 + j) / 2] = (uint8_t)(lo | (hi << 4));
    }
  }
}

/* N(0,1) values of `stream`, indices [0, n), rounded to E4M3. */
void synth_normal_e4m3(uint64_t seed, uint64_t stream, int64_t n, uint8_t* out) {
  int64_t i;
#pragma omp parallel for schedule(static)
  for (i = 0; i < n; i++) out[i] = enc_e4m3(synth_normal(seed, stream, (uint64_t)i));
}

void synth_e4m3_decode(const uint8_t* b, int64_t n, double* out) {
  int64_t i;
  for (i = 0; i < n; i++) out[i] = dec_e4m3(b[i]);
}

void synth_e4m3_encode(const double* x, int64_t n, uint8_t* out) {
  int64_t i;
  for (i = 0; i < n; i++) out[i] = enc_e4m3(x[i]);
}

void synth_nvfp4_encode_rows(const double* x, int64_t nrows, uint8_t* codes, uint8_t* scales) {
  int64_t r;
  for (r = 0; r < nrows; r++) enc_nvfp4_row(x + r * 128, codes + r * 64, scales + r * 8);
}

/*
 * Fill NVFP4 pages. Row (page p, head h, slot s) holds N(0,1) values of
 * `stream` at indices ((p*heads + h)*128 + s)*128 + d. Then, in this order:
 *   - if lognormal_groups: each 16-element group is multiplied by exp(z),
 *     z ~ N(0,1) from stream `stream + 1` at index (row*8 + group);
 *   - if add_index[p] >= 0, the 128-vector add_vecs[add_index[p]] is added
 *     to every valid slot of page p (all heads);
 *   - the row is NVFP4-encoded.
 * Slots s >= page_valid[p] are filled with arbitrary bytes from stream
 * `stream + 2` (they model cache slots not yet written).
 */
void synth_fill_pages(uint64_t seed, uint64_t stream, int64_t num_pages, int heads,
                      const int32_t* page_valid, int lognormal_groups,
                      const int32_t* add_index, const double* add_vecs,
                      uint8_t* codes, uint8_t* scales) {
  int64_t p;
  const uint64_t kx = key_of(seed, stream);
#pragma omp parallel for schedule(dynamic, 4)
  for (p = 0; p < num_pages; p++) {
    int h, s, d, k;
    double x[128];
    for (h = 0; h < heads; h++)
      for (s = 0; s < 128; s++) {
        int64_t row = ((int64_t)p * heads + h) * 128 + s;
        uint8_t* c = codes + row * 64;
        uint8_t* sc = scales + row * 8;
        if (s >= page_valid[p]) {
          for (d = 0; d < 64; d++) c[d] = (uint8_t)(synth_u64(seed, stream + 2, (uint64_t)row * 72 + d) >> 56);
          for (d = 0; d < 8; d++) sc[d] = (uint8_t)(synth_u64(seed, stream + 2, (uint64_t)row * 72 + 64 + d) >> 56);
          continue;
        }
        for (d = 0; d < 128; d += 2) normal_pair(kx, ((uint64_t)row * 128 + d) >> 1, &x[d], &x[d + 1]);
        if (lognormal_groups)
          for (d = 0; d < 8; d++) {
            double f = exp(synth_normal(seed, stream + 1, (uint64_t)row * 8 + d));
            for (k = 0; k < 16; k++) x[d * 16 + k] *= f;
          }
        if (add_index && add_index[p] >= 0)
          for (d = 0; d < 128; d++) x[d] += add_vecs[(int64_t)add_index[p] * 128 + d];
        enc_nvfp4_row(x, c, sc);
      }
  }
}

int synth_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
