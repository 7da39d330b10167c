/* Host side of the seeded input generator, in C with OpenMP: the same values as
 * the numpy definition in synth/__init__.py (checked by tests), fast enough to
 * materialise multi-gigabyte expert weights for the oracle. */
#include <stdint.h>
#include <string.h>

static const uint64_t kGamma = 0x9E3779B97F4A7C15ull;
static const uint64_t kM1 = 0xBF58476D1CE4E5B9ull;
static const uint64_t kM2 = 0x94D049BB133111EBull;
static const uint64_t kField = (1ull << 21) - 1;

static inline uint64_t mix64(uint64_t z) {
  z ^= z >> 30;
  z *= kM1;
  z ^= z >> 27;
  z *= kM2;
  return z ^ (z >> 31);
}

static inline uint16_t bf16_rne(float v) {
  uint32_t b;
  memcpy(&b, &v, 4);
  return (uint16_t)((b + 0x7FFFu + ((b >> 16) & 1u)) >> 16);
}

/* dtype 0: float32 output; 1: bfloat16 bit patterns. */
void synth_host_fill_normal(void* dst, int64_t n, int dtype, uint64_t seed, uint64_t tensor_id, int64_t start,
                            float sigma) {
  const uint64_t key = mix64(seed * kGamma + tensor_id);
  const int64_t bias = 6 * (int64_t)kField;
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    const uint64_t idx = (uint64_t)(start + i);
    int64_t s = 0;
    for (int j = 0; j < 4; ++j) {
      const uint64_t w = mix64(key + (idx * 4ull + (uint64_t)(j + 1)) * kGamma);
      s += (int64_t)(w & kField) + (int64_t)((w >> 21) & kField) + (int64_t)((w >> 42) & kField);
    }
    const float nrm = (float)(s - bias) * 0x1p-21f; /* exact */
    const float v = nrm * sigma;                        /* one IEEE float32 multiply */
    if (dtype == 1)
      ((uint16_t*)dst)[i] = bf16_rne(v);
    else
      ((float*)dst)[i] = v;
  }
}
