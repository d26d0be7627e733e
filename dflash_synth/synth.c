/*
 * Seeded synthetic inputs for the DFlash block drafter: weights, context taps,
 * anchor tokens and a synthetic target's greedy tokens.
 *
 * This file holds no arithmetic of the drafter itself. It is the one module
 * both the CPU oracle's tests and the CUDA path's tests/bench draw inputs
 * from, so both sides see bit-identical inputs.
 *
 * Generator (counter based, so any element can be produced independently of
 * chunking or thread count):
 *   splitmix64(x): z = x + 0x9e3779b97f4a7c15;
 *                  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9;
 *                  z = (z ^ (z >> 27)) * 0x94d049bb133111eb;
 *                  return z ^ (z >> 31)           (Steele, Lea, Flood 2014)
 *   stream key  = splitmix64(seed ^ splitmix64(tensor_id))
 *   uniform(i)  = ((splitmix64(key + i) >> 11) + 0.5) * 2^-53   in (0, 1)
 *   normal(2j), normal(2j+1) = Box-Muller over uniform(2j), uniform(2j+1):
 *                  r = sqrt(-2 ln u1); (r cos 2πu2, r sin 2πu2)
 * Group-64 affine 4-bit quantiser (min/max): for each row and each run of 64
 * inputs, s = bf16((max-min)/15), b = bf16(min), q = clamp(rint((w-b)/s), 0, 15);
 * packed as u32 words, nibble i of word j holding input 8j+i (low nibble first).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define TWO_PI 6.283185307179586476925286766559

static inline uint64_t splitmix64(uint64_t x) {
  uint64_t z = x + 0x9e3779b97f4a7c15ULL;
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ULL;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebULL;
  return z ^ (z >> 31);
}

uint64_t syn_key(uint64_t seed, uint64_t tensor_id) {
  return splitmix64(seed ^ splitmix64(tensor_id));
}

static inline double uniform_at(uint64_t key, uint64_t i) {
  return ((double)(splitmix64(key + i) >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}

static inline double normal_at(uint64_t key, uint64_t i) {
  uint64_t j = i >> 1;
  double u1 = uniform_at(key, 2 * j), u2 = uniform_at(key, 2 * j + 1);
  double r = sqrt(-2.0 * log(u1));
  return (i & 1) ? r * sin(TWO_PI * u2) : r * cos(TWO_PI * u2);
}

/* out[i] = std * normal(offset + i), i < n */
void syn_normal_f32(uint64_t key, uint64_t offset, int64_t n, float std, float* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; i++) out[i] = (float)(std * normal_at(key, offset + (uint64_t)i));
}

void syn_uniform_f64(uint64_t key, uint64_t offset, int64_t n, double* out) {
  for (int64_t i = 0; i < n; i++) out[i] = uniform_at(key, offset + (uint64_t)i);
}

/* tokens uniform in [0, vocab) */
void syn_tokens(uint64_t key, uint64_t offset, int64_t n, int32_t vocab, int32_t* out) {
  for (int64_t i = 0; i < n; i++)
    out[i] = (int32_t)(splitmix64(key + offset + (uint64_t)i) % (uint64_t)vocab);
}

static inline uint16_t bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

static inline float bf16_to_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

void syn_to_bf16(const float* in, int64_t n, uint16_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; i++) out[i] = bf16_rne(in[i]);
}

/* w [rows][cols] fp32 (cols % 64 == 0) -> packed [rows][cols/8] u32,
 * scale/bias [rows][cols/64] bf16 bits. */
void syn_quantize_q4g64(const float* w, int64_t rows, int64_t cols, uint32_t* packed,
                        uint16_t* scale, uint16_t* bias) {
  const int64_t groups = cols / 64;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; r++) {
    for (int64_t g = 0; g < groups; g++) {
      const float* v = w + r * cols + g * 64;
      float mn = v[0], mx = v[0];
      for (int i = 1; i < 64; i++) {
        if (v[i] < mn) mn = v[i];
        if (v[i] > mx) mx = v[i];
      }
      uint16_t sb = bf16_rne((mx - mn) / 15.0f), bb = bf16_rne(mn);
      float s = bf16_to_f32(sb), b = bf16_to_f32(bb);
      scale[r * groups + g] = sb;
      bias[r * groups + g] = bb;
      for (int j = 0; j < 8; j++) {
        uint32_t word = 0;
        for (int i = 0; i < 8; i++) {
          float q = (s > 0.0f) ? rintf((v[8 * j + i] - b) / s) : 0.0f;
          if (q < 0.0f) q = 0.0f;
          if (q > 15.0f) q = 15.0f;
          word |= ((uint32_t)q) << (4 * i);
        }
        packed[r * (cols / 8) + g * 8 + j] = word;
      }
    }
  }
}

/* Synthetic target greedy tokens for one block: t[k] = draft[k] with
 * probability p (k < n), otherwise uniform over the other vocab - 1 tokens;
 * the bonus position t[n] is uniform over the vocabulary. */
void syn_target_tokens(uint64_t key, uint64_t offset, int32_t n, const int32_t* draft, double p,
                       int32_t vocab, int32_t* target) {
  for (int32_t k = 0; k <= n; k++) {
    uint64_t c = offset + 3ull * (uint64_t)k;
    if (k < n) {
      double u = uniform_at(key, c);
      if (u < p) {
        target[k] = draft[k];
      } else {
        uint64_t alt = splitmix64(key + c + 1) % (uint64_t)(vocab - 1);
        target[k] = (int32_t)((draft[k] + 1 + (int64_t)alt) % vocab);
      }
    } else {
      target[k] = (int32_t)(splitmix64(key + c + 2) % (uint64_t)vocab);
    }
  }
}
