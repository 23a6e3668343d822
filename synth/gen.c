/*
 * Seeded synthetic input generator (shared by the CUDA library's tests and
 * benchmark and by the oracle's checks).  It holds none of the method's
 * arithmetic: only a counter-based random generator and the Box-Muller
 * transform.
 *
 * Philox4x32-10: Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
 * easy as 1, 2, 3", SC'11.  Block i (counter words {lo32(i), hi32(i), 0, 0},
 * key {key0, key1}) yields four 32-bit words; the key is bumped by the Weyl
 * constants between rounds.
 */
#include <math.h>
#include <stdint.h>

static void philox_block(uint64_t i, uint32_t k0, uint32_t k1, uint32_t out[4]) {
  uint32_t c0 = (uint32_t)i, c1 = (uint32_t)(i >> 32), c2 = 0, c3 = 0;
  for (int r = 0; r < 10; ++r) {
    uint64_t p0 = (uint64_t)0xD2511F53u * c0;
    uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  out[0] = c0;
  out[1] = c1;
  out[2] = c2;
  out[3] = c3;
}

void synth_philox_words(uint32_t key0, uint32_t key1, uint64_t block0, int64_t nblocks,
                        uint32_t* out) {
  for (int64_t b = 0; b < nblocks; ++b) philox_block(block0 + (uint64_t)b, key0, key1, out + 4 * b);
}

static double u01(uint32_t w) { return ((double)w + 0.5) * (1.0 / 4294967296.0); }

/* Uniform (0,1) stream: element j is word j%4 of block j/4. */
void synth_uniform(uint32_t seed, uint32_t stream, int64_t start, int64_t n, double* out) {
  uint32_t w[4];
  uint64_t cur = (uint64_t)-1;
  for (int64_t j = 0; j < n; ++j) {
    uint64_t e = (uint64_t)(start + j);
    if (e / 4 != cur) {
      cur = e / 4;
      philox_block(cur, seed, stream, w);
    }
    out[j] = u01(w[e % 4]);
  }
}

/* Standard normal stream: block i gives normals 4i..4i+3 by Box-Muller on
 * the word pairs (w0, w1) and (w2, w3). */
static double normal_at(uint64_t e, uint32_t seed, uint32_t stream, uint64_t* cur, double z[4]) {
  if (e / 4 != *cur) {
    uint32_t w[4];
    *cur = e / 4;
    philox_block(*cur, seed, stream, w);
    double r0 = sqrt(-2.0 * log(u01(w[0]))), t0 = 2.0 * M_PI * u01(w[1]);
    double r1 = sqrt(-2.0 * log(u01(w[2]))), t1 = 2.0 * M_PI * u01(w[3]);
    z[0] = r0 * cos(t0);
    z[1] = r0 * sin(t0);
    z[2] = r1 * cos(t1);
    z[3] = r1 * sin(t1);
  }
  return z[e % 4];
}

/* Round a double to bf16 bits through binary32 (nearest-even at both steps). */
static uint16_t to_bf16(double v) {
  float f = (float)v;
  union { float f; uint32_t u; } c = {f};
  if (isnan(f)) return 0x7FC0;
  uint32_t u = c.u;
  return (uint16_t)((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
}

/* bf16 bits of mean + sigma * N(0,1); an element is multiplied by
 * outlier_scale when an independent uniform (stream + 0x10000) falls below
 * outlier_p. */
void synth_bf16_normal(uint32_t seed, uint32_t stream, int64_t start, int64_t n, double mean,
                       double sigma, double outlier_p, double outlier_scale, uint16_t* out) {
  uint64_t cur_n = (uint64_t)-1, cur_u = (uint64_t)-1;
  double z[4], w4[4] = {0, 0, 0, 0};
  uint32_t wu[4];
  for (int64_t j = 0; j < n; ++j) {
    uint64_t e = (uint64_t)(start + j);
    double v = mean + sigma * normal_at(e, seed, stream, &cur_n, z);
    if (outlier_p > 0.0) {
      if (e / 4 != cur_u) {
        cur_u = e / 4;
        philox_block(cur_u, seed, stream + 0x10000u, wu);
        for (int k = 0; k < 4; ++k) w4[k] = u01(wu[k]);
      }
      if (w4[e % 4] < outlier_p) v *= outlier_scale;
    }
    out[j] = to_bf16(v);
  }
}
