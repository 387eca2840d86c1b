// Seeded synthetic inputs for the Stable-LatentMoE routed-expert layer (device side).
//
// Device twin of synth_host.c: the same SplitMix64 streams (Steele, Lea and Flood, OOPSLA
// 2014) and the same value rules, so a tensor filled here is byte-identical to the host
// fill. It holds none of the layer's arithmetic. Used for the K3-sized tensors (15.7 GB of
// MXFP4 experts per layer), which are too large to generate on the host and copy over.
#include <cstdint>
#include <cstddef>
#include <cuda_runtime.h>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ULL;

__host__ __device__ inline uint64_t fmix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}
__host__ __device__ inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
  return fmix64(fmix64(seed + kGamma) ^ stream);
}
__device__ inline uint64_t out64(uint64_t key, uint64_t n) { return fmix64(key + (n + 1) * kGamma); }

__device__ inline uint16_t bf16_rne(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40u);
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

__device__ inline float normal_at(uint64_t key, uint64_t i) {
  long long s = 0;
#pragma unroll
  for (int h = 0; h < 3; ++h) {
    uint64_t r = out64(key, 3 * i + h);
    s += (long long)(r & 0xffff) + (long long)((r >> 16) & 0xffff) +
         (long long)((r >> 32) & 0xffff) + (long long)(r >> 48);
  }
  return __fmul_rn((float)(s - 393210), 1.0f / 65536.0f);
}

__global__ void k_bytes_aligned(uint64_t key, uint64_t word0, size_t nwords, uint64_t* out) {
  for (size_t w = blockIdx.x * (size_t)blockDim.x + threadIdx.x; w < nwords;
       w += (size_t)gridDim.x * blockDim.x)
    out[w] = out64(key, word0 + w);
}

__global__ void k_bytes(uint64_t key, uint64_t offset, size_t n, uint8_t* out) {
  for (size_t j = blockIdx.x * (size_t)blockDim.x + threadIdx.x; j < n;
       j += (size_t)gridDim.x * blockDim.x) {
    uint64_t i = offset + j;
    out[j] = (uint8_t)(out64(key, i >> 3) >> (8 * (i & 7)));
  }
}

__global__ void k_uniform_u8(uint64_t key, uint64_t offset, size_t n, int lo, uint64_t span,
                             uint8_t* out) {
  for (size_t j = blockIdx.x * (size_t)blockDim.x + threadIdx.x; j < n;
       j += (size_t)gridDim.x * blockDim.x) {
    uint64_t r = out64(key, offset + j) >> 32;
    out[j] = (uint8_t)(lo + (int)((r * span) >> 32));
  }
}

__global__ void k_bf16_normal(uint64_t key, uint64_t offset, size_t n, float sigma, uint16_t* out) {
  for (size_t j = blockIdx.x * (size_t)blockDim.x + threadIdx.x; j < n;
       j += (size_t)gridDim.x * blockDim.x)
    out[j] = bf16_rne(__fmul_rn(normal_at(key, offset + j), sigma));
}

inline unsigned grid_for(size_t n) {
  size_t b = (n + 255) / 256;
  if (b > 152u * 32u) b = 152u * 32u;
  return (unsigned)(b == 0 ? 1 : b);
}

}  // namespace

extern "C" {

// All fills: `out` is device memory of n elements, launched on `stream`. Return a
// cudaError_t value (0 = success).
int k3s_dev_fill_bytes(uint64_t seed, uint64_t stream, uint64_t offset, size_t n, void* out,
                       void* cuda_stream) {
  if (n == 0) return 0;
  cudaStream_t s = (cudaStream_t)cuda_stream;
  const uint64_t key = stream_key(seed, stream);
  if ((offset & 7) == 0 && (n & 7) == 0 && ((uintptr_t)out & 7) == 0) {
    k_bytes_aligned<<<grid_for(n / 8), 256, 0, s>>>(key, offset >> 3, n >> 3, (uint64_t*)out);
  } else {
    k_bytes<<<grid_for(n), 256, 0, s>>>(key, offset, n, (uint8_t*)out);
  }
  return (int)cudaGetLastError();
}

int k3s_dev_fill_uniform_u8(uint64_t seed, uint64_t stream, uint64_t offset, size_t n, int lo,
                            int hi, void* out, void* cuda_stream) {
  if (n == 0) return 0;
  k_uniform_u8<<<grid_for(n), 256, 0, (cudaStream_t)cuda_stream>>>(
      stream_key(seed, stream), offset, n, lo, (uint64_t)(hi - lo + 1), (uint8_t*)out);
  return (int)cudaGetLastError();
}

int k3s_dev_fill_bf16_normal(uint64_t seed, uint64_t stream, uint64_t offset, size_t n,
                             float sigma, void* out, void* cuda_stream) {
  if (n == 0) return 0;
  k_bf16_normal<<<grid_for(n), 256, 0, (cudaStream_t)cuda_stream>>>(
      stream_key(seed, stream), offset, n, sigma, (uint16_t*)out);
  return (int)cudaGetLastError();
}

}  // extern "C"
