/* Host implementation of the seeded input generator (see synth.h). Build with
 * -ffp-contract=off so that offset + sigma * z stays two roundings, as on the device. */
#include "synth.h"

#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}
static inline uint64_t splitmix(uint64_t x) { return mix64(x + GOLDEN); }

uint64_t synth_tid(int kind, int layer, int sub) {
  return ((uint64_t)(uint32_t)kind << 32) | ((uint64_t)(uint16_t)layer << 16) | (uint64_t)(uint16_t)sub;
}
uint64_t synth_key(uint64_t seed, uint64_t tid) { return splitmix(splitmix(seed) ^ tid); }
uint64_t synth_draw(uint64_t key, uint64_t n) { return splitmix(key + n * GOLDEN); }

static inline uint32_t sum16(uint64_t r) {
  return (uint32_t)(r & 0xFFFF) + (uint32_t)((r >> 16) & 0xFFFF) + (uint32_t)((r >> 32) & 0xFFFF) +
         (uint32_t)(r >> 48);
}

float synth_normal(uint64_t key, uint64_t i) {
  uint32_t s = sum16(synth_draw(key, 3 * i)) + sum16(synth_draw(key, 3 * i + 1)) +
               sum16(synth_draw(key, 3 * i + 2));
  return (float)((int32_t)s - 393216) * (1.0f / 65536.0f);
}

uint16_t synth_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

void synth_fill_bf16(uint64_t seed, uint64_t tid, uint64_t start, uint64_t count, float sigma,
                     float offset, uint16_t* out) {
  const uint64_t key = synth_key(seed, tid);
  const int with_offset = offset != 0.0f;
#pragma omp parallel for schedule(static) if (count > 65536)
  for (int64_t i = 0; i < (int64_t)count; ++i) {
    float z = synth_normal(key, start + (uint64_t)i);
    float v = sigma * z;
    if (with_offset) v = offset + v;
    out[i] = synth_bf16(v);
  }
}

void synth_fill_uniform_int(uint64_t seed, uint64_t tid, uint64_t start, uint64_t count, int64_t lo,
                            int64_t hi, int64_t* out) {
  const uint64_t key = synth_key(seed, tid);
  const uint64_t span = (uint64_t)(hi - lo + 1);
  for (uint64_t i = 0; i < count; ++i) {
    uint64_t u = synth_draw(key, start + i) >> 32;
    out[i] = lo + (int64_t)((u * span) >> 32);
  }
}

void synth_permutation(uint64_t seed, uint64_t tid, int64_t n, int32_t* out) {
  const uint64_t key = synth_key(seed, tid);
  for (int64_t i = 0; i < n; ++i) out[i] = (int32_t)i;
  for (int64_t i = n - 1; i > 0; --i) {
    uint64_t u = synth_draw(key, (uint64_t)i) >> 32;
    int64_t j = (int64_t)((u * (uint64_t)(i + 1)) >> 32);
    int32_t t = out[i];
    out[i] = out[j];
    out[j] = t;
  }
}
