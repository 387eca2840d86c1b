// Dense bf16 projections for small token counts (decode): router logits, latent in, latent out.
//
//   out[t][n] = sum_k W[n][k] x[t][k]   (fp32 accumulation)
//
// "kimi-k3-mlx", Architecture table: router over 896 experts from the 7168-wide residual;
// Stable LatentMoE: the routed experts see the residual projected to 3584 and their combined
// output is projected back.
//
// HBM-bound: every weight byte is read once. A persistent CTA takes units of 32 weight rows;
// a producer warp streams each unit's rows through a ring of shared-memory stages with
// per-row bulk copies (TMA engine), eight consumer warps split K and run mma.sync bf16 tiles
// (weight rows on M, tokens on N), and a shared-memory reduction in fixed warp order keeps the
// result deterministic. Rows land with a 64-byte pad so the fragment loads are conflict-free.
// Epilogues: fp32 + bias (router logits), bf16 (z, y), and for z also the f16 block-scaled
// copy the expert GEMV reads (one power-of-two exponent per token and 32 features; in MXFP8
// mode the copy holds the MXFP8 round trip of z).
#include <cuda_fp16.h>

#include "k3moe_device.cuh"
#include "k3moe_internal.cuh"

namespace k3moe {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = 32 * (1 + kConsumerWarps);
constexpr int kStages = 3;

struct DenseProblem {
  const uint16_t* W;
  int N;
  float* out_f32;
  const float* bias;
  uint16_t* out_bf16;
  __half* out_h;
  int8_t* out_s;
  int actq;
};

struct DenseArgs {
  DenseProblem p[2];
  int units0, units;  // units of problem 0, total units
  const uint16_t* x;
  int T, K, KC;       // tokens, reduction length, K elements per stage
  uint32_t* err;
};

template <int NTT>
__global__ void __launch_bounds__(kThreads, 1) dense_gemv_kernel(const __grid_constant__ DenseArgs args) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int K = args.K, KC = args.KC, T = args.T;
  const int row_stride = KC * 2 + 64;
  const int stage_bytes = kUnitRows * row_stride;
  const int ntok = 8 * NTT;
  uint8_t* stages = smem;
  float* red = reinterpret_cast<float*>(smem + kStages * stage_bytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(red + kConsumerWarps * kUnitRows * ntok);
  uint64_t* empty = full + kStages;
  uint64_t* cbar = empty + kStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(cbar + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    mbar_init(cbar, 32 * kConsumerWarps);
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  const int nkc = K / KC;
  const int nchunks = (T + ntok - 1) / ntok;

  if (warp == 0) {
    // ---------------- producer
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < args.units && ok; u += gridDim.x) {
      const int pi = u < args.units0 ? 0 : 1;
      const DenseProblem& P = args.p[pi];
      const int row0 = (pi == 0 ? u : u - args.units0) * kUnitRows;
      const int nrows = min(kUnitRows, P.N - row0);
      for (int ch = 0; ch < nchunks && ok; ++ch) {
        for (int kc = 0; kc < nkc; ++kc) {
          if (!mbar_wait_bounded(&empty[s], ph ^ 1, abort_flag, args.err)) { ok = false; break; }
          if (lane == 0) mbar_arrive_expect_tx(&full[s], (uint32_t)(nrows * KC * 2));
          __syncwarp();
          if (lane < nrows)
            bulk_g2s(stages + s * stage_bytes + lane * row_stride,
                     P.W + (size_t)(row0 + lane) * K + (size_t)kc * KC, KC * 2, &full[s]);
          if (++s == kStages) { s = 0; ph ^= 1; }
        }
      }
    }
    if (!ok) {
      // drain: wait (bounded) for copies this warp issued into the stages
      for (int i = 0; i < kStages; ++i) {
        if (--s < 0) { s = kStages - 1; ph ^= 1; }
        volatile int dummy = 0;
        mbar_wait_bounded(&full[s], ph, &dummy, args.err);
      }
    }
    return;
  }

  // ---------------- consumers
  const int cw = warp - 1;
  const int g = lane >> 2, t = lane & 3;
  const int kb_per_stage = KC / 32;
  const int kb_per_warp = (kb_per_stage + kConsumerWarps - 1) / kConsumerWarps;
  int s = 0;
  uint32_t ph = 0, cph = 0;
  for (int u = blockIdx.x; u < args.units; u += gridDim.x) {
    const int pi = u < args.units0 ? 0 : 1;
    const DenseProblem& P = args.p[pi];
    const int row0 = (pi == 0 ? u : u - args.units0) * kUnitRows;
    for (int ch = 0; ch < nchunks; ++ch) {
      const int tok0 = ch * ntok;
      float acc[2][NTT][4];
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int n = 0; n < NTT; ++n)
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[m][n][i] = 0.f;

      for (int kc = 0; kc < nkc; ++kc) {
        if (!mbar_wait_bounded(&full[s], ph, abort_flag, args.err)) return;
        const uint8_t* sb = stages + s * stage_bytes;
        for (int i = 0; i < kb_per_warp; ++i) {
          const int kb = cw * kb_per_warp + i;
          if (kb >= kb_per_stage) break;
          const int kglob = kc * KC + kb * 32 + 8 * t;
          uint4 b[NTT];
#pragma unroll
          for (int n = 0; n < NTT; ++n) {
            const int tok = tok0 + n * 8 + g;
            b[n] = tok < T ? ldg_nc_v4(args.x + (size_t)tok * K + kglob) : make_uint4(0, 0, 0, 0);
          }
#pragma unroll
          for (int m = 0; m < 2; ++m) {
            const uint4 alo = *reinterpret_cast<const uint4*>(sb + (m * 16 + g) * row_stride + kb * 64 + 16 * t);
            const uint4 ahi = *reinterpret_cast<const uint4*>(sb + (m * 16 + g + 8) * row_stride + kb * 64 + 16 * t);
#pragma unroll
            for (int n = 0; n < NTT; ++n) {
              mma_bf16(acc[m][n], alo.x, ahi.x, alo.y, ahi.y, b[n].x, b[n].y);
              mma_bf16(acc[m][n], alo.z, ahi.z, alo.w, ahi.w, b[n].z, b[n].w);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        if (++s == kStages) { s = 0; ph ^= 1; }
      }

      // deterministic cross-warp reduction
      float* r = red + cw * kUnitRows * ntok;
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int n = 0; n < NTT; ++n) {
          r[(m * 16 + g) * ntok + n * 8 + 2 * t] = acc[m][n][0];
          r[(m * 16 + g) * ntok + n * 8 + 2 * t + 1] = acc[m][n][1];
          r[(m * 16 + g + 8) * ntok + n * 8 + 2 * t] = acc[m][n][2];
          r[(m * 16 + g + 8) * ntok + n * 8 + 2 * t + 1] = acc[m][n][3];
        }
      if (!group_barrier(cbar, cph, abort_flag, args.err)) return;
      // epilogue: warp = token, lane = row within the unit
      for (int j = cw; j < ntok; j += kConsumerWarps) {
        const int tok = tok0 + j;
        if (tok >= T) break;
        const int row = row0 + lane;
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) v += red[(w * kUnitRows + lane) * ntok + j];
        const bool valid = row < P.N;
        if (P.out_f32 && valid) P.out_f32[(size_t)tok * P.N + row] = v + (P.bias ? P.bias[row] : 0.f);
        if (P.out_bf16) {
          const uint16_t vb = f32_to_bf16(v);
          if (valid) P.out_bf16[(size_t)tok * P.N + row] = vb;
          if (P.out_h) {  // N is a multiple of 32 here: the whole warp is one block
            float q = bf16_to_f32(vb);
            if (P.actq) q = mxfp8_roundtrip(q, mxfp8_block_exp(warp_max(fabsf(q))));
            const int e = f16_block_exp(warp_max(fabsf(q)));
            P.out_h[(size_t)tok * P.N + row] = __float2half_rn(ldexpf(q, -e));
            if (lane == 0) P.out_s[(size_t)tok * (P.N / 32) + row0 / 32] = (int8_t)e;
          }
        }
      }
      if (!group_barrier(cbar, cph, abort_flag, args.err)) return;
    }
  }
}

template <int NTT>
cudaError_t launch_t(const DenseArgs& a, cudaStream_t s) {
  const int row_stride = a.KC * 2 + 64;
  const size_t smem = (size_t)kStages * kUnitRows * row_stride +
                      (size_t)kConsumerWarps * kUnitRows * 8 * NTT * sizeof(float) +
                      (2 * kStages + 1) * sizeof(uint64_t) + 16;
  cudaError_t e = cudaFuncSetAttribute(dense_gemv_kernel<NTT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int grid = a.units < num_sms() ? a.units : num_sms();
  dense_gemv_kernel<NTT><<<grid, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dense_gemv(const uint16_t* W0, int N0, float* out0_f32, uint16_t* out0_bf16,
                              const float* bias0, const uint16_t* W1, int N1, uint16_t* out1_bf16,
                              __half* out1_h, int8_t* out1_s, int actq1, const uint16_t* x, int T,
                              int K, uint32_t* err, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  DenseArgs a{};
  a.p[0] = DenseProblem{W0, N0, out0_f32, bias0, out0_bf16, nullptr, nullptr, 0};
  a.p[1] = DenseProblem{W1, N1, nullptr, nullptr, out1_bf16, out1_h, out1_s, actq1};
  a.units0 = W0 ? (N0 + kUnitRows - 1) / kUnitRows : 0;
  a.units = a.units0 + (W1 ? (N1 + kUnitRows - 1) / kUnitRows : 0);
  a.x = x;
  a.T = T;
  a.K = K;
  a.KC = (K % 512 == 0) ? 512 : (K % 256 == 0) ? 256 : (K % 128 == 0) ? 128 : 64;
  a.err = err;
  if (a.units == 0) return cudaSuccess;
  if (T <= 8) return launch_t<1>(a, s);
  if (T <= 16) return launch_t<2>(a, s);
  if (T <= 32) return launch_t<4>(a, s);
  return launch_t<8>(a, s);
}

}  // namespace k3moe
