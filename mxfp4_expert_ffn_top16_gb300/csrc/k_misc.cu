// Small elementwise kernels: the routing-weighted combine, and the f16 block-scaled
// activation copy the expert GEMV reads.
#include <cuda_fp16.h>

#include "k3moe_device.cuh"
#include "k3moe_internal.cuh"

namespace k3moe {
namespace {

// c[t][n] = bf16(sum_{j<k} w[t][j] * o[slot_row[t*k+j]][n]), fp32, j ascending.
// Routed outputs are combined in latent space before the projection back to the residual
// ("kimi-k3-mlx", LatentMoE).
// Two values per thread; the k rows and weights are loaded before any is summed, so all of a
// thread's loads are in flight together (few tokens leave this kernel latency-bound).
constexpr int kMaxTopK = 32;
__global__ void combine_kernel(const float* __restrict__ o, const int32_t* __restrict__ slot_row,
                               const float* __restrict__ w, int T, int k, int L, uint16_t* c) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.y;
  const int n = (blockIdx.x * blockDim.x + threadIdx.x) * 2;
  if (t >= T || n >= L) return;
  int rr[kMaxTopK];
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) rr[j] = j < k ? slot_row[(size_t)t * k + j] : -1;
  float2 v[kMaxTopK];
  float wj[kMaxTopK];
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    const bool ok = j < k && rr[j] >= 0 && rr[j] < T * k;  // out-of-range rows contribute nothing
    v[j] = ok ? *reinterpret_cast<const float2*>(o + (size_t)rr[j] * L + n) : make_float2(0.f, 0.f);
    wj[j] = ok ? w[(size_t)t * k + j] : 0.f;
    if (!ok) rr[j] = -1;
  }
  // Kahan-compensated sum in slot order, so the bf16 rounding of c follows the exact sum of
  // the fp32 terms except within ~1 fp32 ulp of a rounding boundary
  float s[2] = {0.f, 0.f}, cc[2] = {0.f, 0.f};
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    if (rr[j] < 0) continue;
    const float p[2] = {wj[j] * v[j].x, wj[j] * v[j].y};
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const float yk = p[q] - cc[q];
      const float tk = s[q] + yk;
      cc[q] = (tk - s[q]) - yk;
      s[q] = tk;
    }
  }
  const uint32_t packed = (uint32_t)f32_to_bf16(s[0] - cc[0]) | ((uint32_t)f32_to_bf16(s[1] - cc[1]) << 16);
  *reinterpret_cast<uint32_t*>(c + (size_t)t * L + n) = packed;
}

// One warp per (token, block of 32 values): optional MXFP8 round trip, then an f16 copy
// scaled by 2^-e with e chosen from the block maximum, and the exponent e.
__global__ void act_prep_kernel(const uint16_t* __restrict__ z, int T, int L, int actq, __half* zh,
                                int8_t* zs) {
  const int lane = threadIdx.x & 31;
  const long long blk = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const long long nblk = (long long)T * (L / 32);
  if (blk >= nblk) return;
  const size_t i = (size_t)blk * 32 + lane;
  float q = bf16_to_f32(z[i]);
  if (actq) q = mxfp8_roundtrip(q, mxfp8_block_exp(warp_max(fabsf(q))));
  const int e = f16_block_exp(warp_max(fabsf(q)));
  zh[i] = __float2half_rn(ldexpf(q, -e));
  if (lane == 0) {
    const long long t = blk / (L / 32), b = blk % (L / 32);
    zs[t * exp_pitch(L) + b] = (int8_t)e;
  }
}

}  // namespace

cudaError_t launch_combine(const float* o_rows, const int32_t* slot_row, const float* w, int T,
                           int k, int L, uint16_t* c, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  if (k > kMaxTopK) return cudaErrorInvalidValue;
  dim3 grid((L / 2 + 127) / 128, T);
  return launch_pdl(combine_kernel, grid, dim3(128), 0, s, o_rows, slot_row, w, T, k, L, c);
}

cudaError_t launch_act_prep(const uint16_t* z, int T, int L, int actq, __half* zh, int8_t* zs,
                            cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  const long long nblk = (long long)T * (L / 32);
  const int warps = 8;
  act_prep_kernel<<<(unsigned)((nblk + warps - 1) / warps), 32 * warps, 0, s>>>(z, T, L, actq, zh, zs);
  return cudaGetLastError();
}

}  // namespace k3moe
