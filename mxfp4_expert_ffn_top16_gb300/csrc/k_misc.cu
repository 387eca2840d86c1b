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
// Four values per thread (16-byte loads); the k rows and weights are loaded before any is
// summed, so all of a thread's loads are in flight together: HBM-bound for many tokens (the
// fp32 rows are read once, with the streaming hint), latency-bound for a few. KB >= k bounds the
// unrolled slot loop.
constexpr int kMaxTopK = 32;
constexpr int kCombineThreads = 128;
template <int KB>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const float* __restrict__ o,
                                                                  const int32_t* __restrict__ slot_row,
                                                                  const float* __restrict__ w, int T, int k,
                                                                  int L, uint16_t* c) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.y;
  const int n = (blockIdx.x * kCombineThreads + threadIdx.x) * 4;
  if (t >= T || n >= L) return;
  int rr[KB];
#pragma unroll
  for (int j = 0; j < KB; ++j) {
    rr[j] = j < k ? __ldg(slot_row + (size_t)t * k + j) : -1;
    if (rr[j] >= T * k) rr[j] = -1;  // out-of-range rows contribute nothing
  }
  float4 v[KB];
  float wj[KB];
#pragma unroll
  for (int j = 0; j < KB; ++j) {
    const bool ok = rr[j] >= 0;
    v[j] = ok ? __ldcs(reinterpret_cast<const float4*>(o + (size_t)rr[j] * L + n)) : make_float4(0.f, 0.f, 0.f, 0.f);
    wj[j] = ok ? __ldg(w + (size_t)t * k + j) : 0.f;
  }
  // Kahan-compensated sum in slot order, so the bf16 rounding of c follows the exact sum of
  // the fp32 terms except within ~1 fp32 ulp of a rounding boundary
  float s[4] = {0.f, 0.f, 0.f, 0.f}, cc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int j = 0; j < KB; ++j) {
    if (rr[j] < 0) continue;
    combine_term(s[0], cc[0], wj[j], v[j].x);
    combine_term(s[1], cc[1], wj[j], v[j].y);
    combine_term(s[2], cc[2], wj[j], v[j].z);
    combine_term(s[3], cc[3], wj[j], v[j].w);
  }
  uint2 packed;
  packed.x = (uint32_t)combine_result(s[0], cc[0]) | ((uint32_t)combine_result(s[1], cc[1]) << 16);
  packed.y = (uint32_t)combine_result(s[2], cc[2]) | ((uint32_t)combine_result(s[3], cc[3]) << 16);
  *reinterpret_cast<uint2*>(c + (size_t)t * L + n) = packed;
}

// Shared experts' GLU: a = bf16(silu(g) * up), silu(g) = g / (1 + e^-g) in the same fast forms
// as the routed experts' epilogue (~1e-6 relative, far below the bf16 rounding). Four
// elements per thread (16-byte loads); n is a multiple of 4.
__global__ void glu_kernel(const float4* __restrict__ g, const float4* __restrict__ u, long long n4,
                           uint2* __restrict__ a) {
  pdl_wait();
  pdl_trigger();
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (long long)gridDim.x * blockDim.x) {
    const float4 gv = g[i], uv = u[i];
    const float gg[4] = {gv.x, gv.y, gv.z, gv.w}, uu[4] = {uv.x, uv.y, uv.z, uv.w};
    uint32_t b[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) b[q] = f32_to_bf16(__fdividef(gg[q], 1.0f + __expf(-gg[q])) * uu[q]);
    a[i] = make_uint2(b[0] | (b[1] << 16), b[2] | (b[3] << 16));
  }
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

// REAP saliency ("kimi-k3-mlx" digest, REAP pruning section: S_j = (1/|C|) sum_x g_j(x)
// ||e_j(x)||_2): one warp per sorted row r (token t, slot j, expert e = idx[t][j]) adds
// w[t][j] * ||o[r]||_2 to S[e]. The squares are summed in fp32 (four per lane per 16-byte load,
// then across the warp), the product and the sum over rows in fp64 (atomic adds, in no fixed
// order).
__global__ void __launch_bounds__(256) saliency_kernel(const float* __restrict__ o, const int32_t* __restrict__ row_token,
                                                       const int32_t* __restrict__ row_slot,
                                                       const int32_t* __restrict__ idx, const float* __restrict__ w,
                                                       int rows, int T, int k, int L, int E, double* S, uint32_t* err) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const long long nw = ((long long)gridDim.x * blockDim.x) >> 5;
  for (long long r = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows; r += nw) {
    const float4* row = reinterpret_cast<const float4*>(o + (size_t)r * L);
    float ss = 0.f;
    for (int n = lane; n < L / 4; n += 32) {
      const float4 v = __ldcs(row + n);
      ss = fmaf(v.x, v.x, ss);
      ss = fmaf(v.y, v.y, ss);
      ss = fmaf(v.z, v.z, ss);
      ss = fmaf(v.w, v.w, ss);
    }
#pragma unroll
    for (int x = 16; x > 0; x >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, x);
    if (lane == 0) {
      const int t = row_token[r], j = row_slot[r];
      const int e = (t >= 0 && t < T && j >= 0 && j < k) ? idx[(size_t)t * k + j] : -1;
      if (e < 0 || e >= E) {
        atomicOr(err, kErrIndex);
      } else {
        atomicAdd(S + e, (double)w[(size_t)t * k + j] * sqrt((double)ss));
      }
    }
  }
}

// 16-byte copy, one launch in the programmatic-launch chain (the host-buffer layer call's token
// read and output write).
// Four 16-byte loads in flight per thread before their stores: the reads cross the CPU-GPU link
// (or the writes do), whose latency a single load per thread would expose.
__global__ void copy16_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, long long n) {
  pdl_wait();
  pdl_trigger();
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += 4 * stride) {
    uint4 v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (i + j * stride < n) v[j] = src[i + j * stride];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (i + j * stride < n) dst[i + j * stride] = v[j];
  }
}

}  // namespace

cudaError_t launch_saliency(const float* o_rows, const int32_t* row_token, const int32_t* row_slot,
                            const int32_t* idx, const float* w, int T, int k, int L, int E, double* S,
                            uint32_t* err, cudaStream_t s) {
  const long long rows = (long long)T * k;
  if (rows <= 0) return cudaSuccess;
  if (L % 4) return cudaErrorInvalidValue;
  long long blocks = (rows + 7) / 8;
  if (blocks > 16LL * num_sms()) blocks = 16LL * num_sms();
  return launch_pdl(saliency_kernel, dim3((unsigned)blocks), dim3(256), 0, s, o_rows, row_token, row_slot, idx, w,
                    (int)rows, T, k, L, E, S, err);
}

cudaError_t launch_combine(const float* o_rows, const int32_t* slot_row, const float* w, int T,
                           int k, int L, uint16_t* c, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  if (k > kMaxTopK || L % 4) return cudaErrorInvalidValue;
  dim3 grid((L / 4 + kCombineThreads - 1) / kCombineThreads, T);
  if (k <= 16)
    return launch_pdl(combine_kernel<16>, grid, dim3(kCombineThreads), 0, s, o_rows, slot_row, w, T, k, L, c);
  return launch_pdl(combine_kernel<kMaxTopK>, grid, dim3(kCombineThreads), 0, s, o_rows, slot_row, w, T, k, L, c);
}

cudaError_t launch_glu(const float* g, const float* u, long long n, uint16_t* a, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  if (n % 4) return cudaErrorInvalidValue;
  const long long n4 = n / 4;
  long long blocks = (n4 + 255) / 256;
  if (blocks > 16LL * num_sms()) blocks = 16LL * num_sms();
  return launch_pdl(glu_kernel, dim3((unsigned)blocks), dim3(256), 0, s, reinterpret_cast<const float4*>(g),
                    reinterpret_cast<const float4*>(u), n4, reinterpret_cast<uint2*>(a));
}

cudaError_t launch_act_prep(const uint16_t* z, int T, int L, int actq, __half* zh, int8_t* zs,
                            cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  const long long nblk = (long long)T * (L / 32);
  const int warps = 8;
  act_prep_kernel<<<(unsigned)((nblk + warps - 1) / warps), 32 * warps, 0, s>>>(z, T, L, actq, zh, zs);
  return cudaGetLastError();
}

cudaError_t launch_copy16(const void* src, void* dst, size_t bytes, cudaStream_t s) {
  const long long n = (long long)(bytes / 16);
  if (n == 0) return cudaSuccess;
  const long long blocks = (n + 255) / 256;
  return launch_pdl(copy16_kernel, dim3((unsigned)(blocks < 2048 ? blocks : 2048)), dim3(256), 0, s,
                    static_cast<const uint4*>(src), static_cast<uint4*>(dst), n);
}

}  // namespace k3moe
