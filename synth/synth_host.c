/*
 * Seeded synthetic inputs for the Stable-LatentMoE routed-expert layer (host side).
 *
 * This file holds no arithmetic of the layer itself: it only turns (seed, stream, index)
 * into input values. The device twin in synth_dev.cu implements the same definitions so
 * that a tensor generated on the GPU and one generated here are byte-identical.
 *
 * Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
 * generators", OOPSLA 2014). Output n of a generator seeded with `key` is
 * fmix(key + (n + 1) * 0x9E3779B97F4A7C15), fmix being the published finaliser below.
 * Every tensor draws from its own stream key = fmix(fmix(seed) ^ stream).
 *
 * Value rules (element i of a tensor):
 *   bytes   : byte (i & 7), little-endian, of output (i >> 3)         -> U{0..255}
 *             (two e2m1 codes per byte, so every code is U{0..15})
 *   uniform : lo + ((output(i) >> 32) * span >> 32), span = hi - lo + 1
 *   normal  : Irwin-Hall sum of 12 uniforms. The twelve 16-bit fields u_j of outputs
 *             3i, 3i+1, 3i+2 give S = sum u_j; v = (S - 393210) * 2^-16, which is
 *             sum_j (u_j + 0.5)/65536 - 6: mean 0, variance 1 (up to the 16-bit grid).
 *             The integer is exact in fp32; the value is then multiplied by sigma in
 *             fp32 and rounded to bf16 (round to nearest even).
 * All steps are integer or single correctly rounded fp32 operations, so host and device
 * agree bit for bit.
 */
#include <stdint.h>
#include <stddef.h>
#include <string.h>

#define K3S_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t fmix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

uint64_t k3s_key(uint64_t seed, uint64_t stream) {
  return fmix64(fmix64(seed + K3S_GAMMA) ^ stream);
}

static inline uint64_t out64(uint64_t key, uint64_t n) {
  return fmix64(key + (n + 1) * K3S_GAMMA);
}

uint64_t k3s_rand64(uint64_t seed, uint64_t stream, uint64_t n) {
  return out64(k3s_key(seed, stream), n);
}

static inline uint16_t bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40u);
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

static inline float normal_at(uint64_t key, uint64_t i) {
  int64_t s = 0;
  for (int h = 0; h < 3; ++h) {
    uint64_t r = out64(key, 3 * i + (uint64_t)h);
    s += (int64_t)(r & 0xffff) + (int64_t)((r >> 16) & 0xffff) +
         (int64_t)((r >> 32) & 0xffff) + (int64_t)(r >> 48);
  }
  volatile float v = (float)(s - 393210) * (1.0f / 65536.0f);
  return v;
}

void k3s_fill_bytes(uint64_t seed, uint64_t stream, uint64_t offset, size_t n, uint8_t* out) {
  const uint64_t key = k3s_key(seed, stream);
  size_t j = 0;
  while (j < n) {
    uint64_t i = offset + j;
    uint64_t r = out64(key, i >> 3);
    out[j++] = (uint8_t)(r >> (8 * (i & 7)));
  }
}

void k3s_fill_uniform_u8(uint64_t seed, uint64_t stream, uint64_t offset, size_t n,
                         int lo, int hi, uint8_t* out) {
  const uint64_t key = k3s_key(seed, stream);
  const uint64_t span = (uint64_t)(hi - lo + 1);
  for (size_t j = 0; j < n; ++j) {
    uint64_t r = out64(key, offset + j) >> 32;
    out[j] = (uint8_t)(lo + (int)((r * span) >> 32));
  }
}

void k3s_fill_uniform_i32(uint64_t seed, uint64_t stream, uint64_t offset, size_t n,
                          int64_t lo, int64_t hi, int32_t* out) {
  const uint64_t key = k3s_key(seed, stream);
  const uint64_t span = (uint64_t)(hi - lo + 1);
  for (size_t j = 0; j < n; ++j) {
    uint64_t r = out64(key, offset + j) >> 32;
    out[j] = (int32_t)(lo + (int64_t)((r * span) >> 32));
  }
}

void k3s_fill_bf16_normal(uint64_t seed, uint64_t stream, uint64_t offset, size_t n,
                          float sigma, uint16_t* out) {
  const uint64_t key = k3s_key(seed, stream);
  for (size_t j = 0; j < n; ++j) {
    volatile float v = normal_at(key, offset + j) * sigma;
    out[j] = bf16_rne(v);
  }
}

void k3s_fill_f32_normal(uint64_t seed, uint64_t stream, uint64_t offset, size_t n,
                         float sigma, float* out) {
  const uint64_t key = k3s_key(seed, stream);
  for (size_t j = 0; j < n; ++j) {
    volatile float v = normal_at(key, offset + j) * sigma;
    out[j] = v;
  }
}
