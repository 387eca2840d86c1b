// Dense bf16 projections for small token counts (decode): router logits, latent in, latent out.
//
//   out[t][n] = sum_k W[n][k] x[t][k]   (fp32 accumulation)
//
// "kimi-k3-mlx", Architecture table: router over 896 experts from the 7168-wide residual;
// Stable LatentMoE: the routed experts see the residual projected to 3584 and their combined
// output is projected back.
//
// HBM-bound: every weight byte is read once per chunk of up to 64 tokens. A persistent CTA
// takes units of 32 weight rows; a producer warp streams, per stage, NB tiles of the unit's
// rows (32 rows x 64 bf16 = 4 KB each) and the matching tiles of the chunk's token rows
// through the TMA engine (2-D tensor maps, 128-byte swizzle) into a ring of shared-memory
// stages; eight consumer warps split K and run mma.sync bf16 tiles (weight rows on M, tokens
// on N). Each 32-wide K block is accumulated in a fresh tile and then added in IEEE fp32, so
// the result does not inherit the tensor core's internal accumulation over the whole of K.
// A shared-memory reduction in fixed warp order keeps the result deterministic.
// Fragment row g of an mma tile reads tile row pi(g) = (g >> 1) | ((g & 1) << 2): with the
// 128-byte swizzle, the rows read in one shared-memory phase then hit disjoint banks.
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
constexpr int kMaxStages = 4;

struct DenseProblem {
  int N;
  float* out_f32;
  const float* bias;
  uint16_t* out_bf16;
  __half* out_h;
  int8_t* out_s;
  int actq;
  uint8_t* out_q;   // optional: the bf16 outputs as qP E4M3 rows per token [T][qP][N] ...
  uint8_t* out_qs;  // ... with e8m0 block exponents [T][qP][exp_pitch(N)]
  int qP;           // 1: MXFP8; 2: bf16 split exactly into hi + lo
};

struct DenseArgs {
  CUtensorMap tw[2];   // W of each problem: {K, N} bf16, box {64, 32}, 128-byte swizzle
  CUtensorMap tx;      // tokens: {K, T} bf16, box {64, 8*NTT}, 128-byte swizzle
  DenseProblem p[2];
  int units0, units;   // units of problem 0, total units
  int T, K, NB, NS;    // tokens, reduction length, tiles per stage along K, stages
  // optional second K segment of problem 0 (a single problem): out = W x + W2 x2; its nkc1
  // K steps follow the first K / (64 NB)
  CUtensorMap tw2, tx2;
  int nkc1;
  int* zero;           // optional: cleared after the grid dependency wait
  int nzero;
  uint32_t* err;
};

__device__ __forceinline__ int pi8(int g) { return (g >> 1) | ((g & 1) << 2); }

template <int NTT>
__global__ void __launch_bounds__(kThreads, 1) dense_gemv_kernel(const __grid_constant__ DenseArgs args) {
  constexpr int ntok = 8 * NTT;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int K = args.K, NB = args.NB, NS = args.NS, T = args.T;
  const int wbox = kUnitRows * 128, xbox = ntok * 128;
  const int stage_bytes = NB * (wbox + xbox);
  uint8_t* stages = smem + ((1024u - (smem_u32(smem) & 1023u)) & 1023u);
  float* red = reinterpret_cast<float*>(stages + NS * stage_bytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(red + kConsumerWarps * kUnitRows * ntok);
  uint64_t* empty = full + kMaxStages;
  uint64_t* cbar = empty + kMaxStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(cbar + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    mbar_init(cbar, kConsumerWarps);
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  const int KC = 64 * NB;
  const int nkc0 = K / KC, nkc = nkc0 + args.nkc1;
  const int nchunks = (T + ntok - 1) / ntok;
  // No earlier kernel writes the weights: the loading thread sends the first stages' weight
  // tiles out before the grid dependency wait, while the kernel before this one finishes (its
  // token tiles, which that kernel may write, follow after the wait).
  const int npre = blockIdx.x < args.units ? (NS < nkc0 ? NS : nkc0) : 0;
  if (threadIdx.x == 0) {
    const int u = blockIdx.x, pi = u < args.units0 ? 0 : 1;
    const int row0 = (pi == 0 ? u : u - args.units0) * kUnitRows;
    const uint64_t pol = l2_evict_first();
    for (int kc = 0; kc < npre; ++kc) {
      mbar_arrive_expect_tx(&full[kc], (uint32_t)stage_bytes);
      tma_load_3d_stream(stages + kc * stage_bytes, &args.tw[pi], 0, row0, kc * NB, &full[kc], pol);
    }
  }
  pdl_wait();
  pdl_trigger();
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < args.nzero; i += blockDim.x) args.zero[i] = 0;

  if (warp == 0) {
    // ---------------- producer (lane 0 issues)
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    const uint64_t pol = l2_evict_first();
    for (int u = blockIdx.x; u < args.units && ok; u += gridDim.x) {
      const int pi = u < args.units0 ? 0 : 1;
      const int row0 = (pi == 0 ? u : u - args.units0) * kUnitRows;
      for (int ch = 0; ch < nchunks && ok; ++ch) {
        for (int kc = 0; kc < nkc; ++kc) {
          if (!mbar_wait_bounded(&empty[s], ph ^ 1, abort_flag, args.err)) { ok = false; break; }
          if (lane == 0) {  // one copy for the NB weight tiles, one for the NB token tiles
            uint8_t* dst = stages + s * stage_bytes;
            const bool seg2 = kc >= nkc0;  // second K segment (problem 0 only)
            if (u != (int)blockIdx.x || ch != 0 || kc >= npre) {  // (else sent before the wait)
              mbar_arrive_expect_tx(&full[s], (uint32_t)stage_bytes);
              tma_load_3d_stream(dst, seg2 ? &args.tw2 : &args.tw[pi], 0, row0, (seg2 ? kc - nkc0 : kc) * NB,
                                 &full[s], pol);
            }
            tma_load_3d(dst + NB * wbox, seg2 ? &args.tx2 : &args.tx, 0, ch * ntok, (seg2 ? kc - nkc0 : kc) * NB,
                        &full[s]);
          }
          __syncwarp();
          if (++s == NS) { s = 0; ph ^= 1; }
        }
      }
    }
    if (!ok) {
      for (int i = 0; i < NS; ++i) {
        if (--s < 0) { s = NS - 1; ph ^= 1; }
        volatile int dummy = 0;
        mbar_wait_bounded(&full[s], ph, &dummy, args.err);
      }
    }
    return;
  }

  // ---------------- consumers
  const int cw = warp - 1;
  const int g = lane >> 2, t = lane & 3;
  const int pg = pi8(g);
  const int kb_per_stage = 2 * NB;  // 32-wide K blocks per stage
  const int kb_per_warp = (kb_per_stage + kConsumerWarps - 1) / kConsumerWarps;
  int s = 0;
  uint32_t ph = 0, cph = 0;
  for (int u = blockIdx.x; u < args.units; u += gridDim.x) {
    const int pi = u < args.units0 ? 0 : 1;
    const DenseProblem& P = args.p[pi];
    const int row0 = (pi == 0 ? u : u - args.units0) * kUnitRows;
    for (int ch = 0; ch < nchunks; ++ch) {
      const int tok0 = ch * ntok;
      // Kahan-compensated sums of the per-block tiles: bf16 rounding of the result (z, y)
      // then depends on the exact sum except within ~1 fp32 ulp of a rounding boundary
      float acc[2][NTT][4], cmp[2][NTT][4];
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int n = 0; n < NTT; ++n)
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[m][n][i] = cmp[m][n][i] = 0.f;

      for (int kc = 0; kc < nkc; ++kc) {
        if (!mbar_wait_bounded(&full[s], ph, abort_flag, args.err)) return;
        const uint8_t* sb = stages + s * stage_bytes;
        for (int i = 0; i < kb_per_warp; ++i) {
          const int kb = cw * kb_per_warp + i;
          if (kb >= kb_per_stage) break;
          const int box = kb >> 1;
          const int col = ((kb & 1) * 4 + t) * 16;  // byte column of this lane's 8 elements
          const uint8_t* wb = sb + box * wbox;
          const uint8_t* xb = sb + NB * wbox + box * xbox;
          uint4 b[NTT];
#pragma unroll
          for (int n = 0; n < NTT; ++n)
            b[n] = *reinterpret_cast<const uint4*>(xb + swz128(n * 8 + pg, col));
#pragma unroll
          for (int m = 0; m < 2; ++m) {
            const uint4 alo = *reinterpret_cast<const uint4*>(wb + swz128(m * 16 + pg, col));
            const uint4 ahi = *reinterpret_cast<const uint4*>(wb + swz128(m * 16 + pg + 8, col));
#pragma unroll
            for (int n = 0; n < NTT; ++n) {
              float tmp[4] = {0.f, 0.f, 0.f, 0.f};
              mma_bf16(tmp, alo.x, ahi.x, alo.y, ahi.y, b[n].x, b[n].y);
              mma_bf16(tmp, alo.z, ahi.z, alo.w, ahi.w, b[n].z, b[n].w);
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const float yk = tmp[q] - cmp[m][n][q];
                const float tk = acc[m][n][q] + yk;
                cmp[m][n][q] = (tk - acc[m][n][q]) - yk;
                acc[m][n][q] = tk;
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        if (++s == NS) { s = 0; ph ^= 1; }
      }

      // deterministic cross-warp reduction; red[w][weight row][token], physical indices
      float* r = red + cw * kUnitRows * ntok;
      const int c0 = pi8(2 * t), c1 = pi8(2 * t + 1);
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int n = 0; n < NTT; ++n) {
          r[(m * 16 + pg) * ntok + n * 8 + c0] = acc[m][n][0] - cmp[m][n][0];
          r[(m * 16 + pg) * ntok + n * 8 + c1] = acc[m][n][1] - cmp[m][n][1];
          r[(m * 16 + pg + 8) * ntok + n * 8 + c0] = acc[m][n][2] - cmp[m][n][2];
          r[(m * 16 + pg + 8) * ntok + n * 8 + c1] = acc[m][n][3] - cmp[m][n][3];
        }
      if (!group_barrier(cbar, cph, abort_flag, args.err)) return;
      // epilogue: warp = token, lane = row within the unit
      for (int j = cw; j < ntok; j += kConsumerWarps) {
        const int tok = tok0 + j;
        if (tok >= T) break;
        const int row = row0 + lane;
        float v = 0.f, vc = 0.f;  // Kahan over the warps' partials, fixed order
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
          const float yk = red[(w * kUnitRows + lane) * ntok + j] - vc;
          const float tk = v + yk;
          vc = (tk - v) - yk;
          v = tk;
        }
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
            if (lane == 0) P.out_s[(size_t)tok * exp_pitch(P.N) + row0 / 32] = (int8_t)e;
          }
          if (P.out_q) {  // the same blocks of 32 features, as E4M3 rows for the tensor cores
            const float q = bf16_to_f32(vb);
            const int sp = exp_pitch(P.N);
            const size_t qr = (size_t)tok * P.qP;
            const int X0 = P.qP == 1 ? mxfp8_block_exp(warp_max(fabsf(q))) : split_block_exp(warp_max(fabsf(q)));
            const uint32_t c0 = e4m3x2(mul_pow2(q, -X0), 0.f) & 0xffu;
            P.out_q[qr * P.N + row] = (uint8_t)c0;
            if (lane == 0) P.out_qs[qr * sp + row0 / 32] = (uint8_t)(X0 + 127);
            if (P.qP == 2) {  // lo = the exact remainder v - hi, on its own block exponent
              const float rem = q - mul_pow2(e4m3x2_value(c0).x, X0);
              const int X1 = split_block_exp(warp_max(fabsf(rem)));
              P.out_q[(qr + 1) * P.N + row] = (uint8_t)(e4m3x2(mul_pow2(rem, -X1), 0.f) & 0xffu);
              if (lane == 0) P.out_qs[(qr + 1) * sp + row0 / 32] = (uint8_t)(X1 + 127);
            }
          }
        }
      }
      if (!group_barrier(cbar, cph, abort_flag, args.err)) return;
    }
  }
}

template <int NTT>
cudaError_t launch_t(DenseArgs& a, const uint16_t* const W[2], const int N[2], const uint16_t* x,
                     const uint16_t* W2, const uint16_t* x2, int K2, cudaStream_t s) {
  constexpr int ntok = 8 * NTT;
  const int target_nb = NTT <= 2 ? 8 : (NTT == 4 ? 4 : 2);
  const int kt = a.K / 64, kt2 = K2 / 64;
  a.NB = 1;
  for (int nb = target_nb; nb >= 1; nb >>= 1)
    if (kt % nb == 0 && kt2 % nb == 0) { a.NB = nb; break; }
  a.nkc1 = kt2 / a.NB;
  if (kt2 > 0 && (!make_tmap_3d_chunks(&a.tw2, W2, 2, 64, (uint64_t)N[0], (uint64_t)K2 * 2, (uint64_t)kt2,
                                       kUnitRows, (uint32_t)a.NB, true) ||
                  !make_tmap_3d_chunks(&a.tx2, x2, 2, 64, (uint64_t)a.T, (uint64_t)K2 * 2, (uint64_t)kt2, ntok,
                                       (uint32_t)a.NB, true)))
    return cudaErrorInvalidValue;
  const int stage_bytes = a.NB * (kUnitRows * 128 + ntok * 128);
  a.NS = NTT <= 2 ? 3 : 4;
  for (int i = 0; i < 2; ++i)
    if (W[i] && !make_tmap_3d_chunks(&a.tw[i], W[i], 2, 64, (uint64_t)N[i], (uint64_t)a.K * 2,
                                     (uint64_t)kt, kUnitRows, (uint32_t)a.NB, true))
      return cudaErrorInvalidValue;
  if (!make_tmap_3d_chunks(&a.tx, x, 2, 64, (uint64_t)a.T, (uint64_t)a.K * 2, (uint64_t)kt, ntok,
                           (uint32_t)a.NB, true))
    return cudaErrorInvalidValue;
  const size_t smem = (size_t)a.NS * stage_bytes + (size_t)kConsumerWarps * kUnitRows * ntok * sizeof(float) +
                      (2 * kMaxStages + 1) * sizeof(uint64_t) + 16 + 1024;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(dense_gemv_kernel<NTT>), smem);
  if (e != cudaSuccess) return e;
  const int grid = a.units < num_sms() ? a.units : num_sms();
  return launch_pdl(dense_gemv_kernel<NTT>, dim3(grid), dim3(kThreads), smem, s, a);
}

}  // namespace

cudaError_t launch_dense_gemv(const uint16_t* W0, int N0, float* out0_f32, uint16_t* out0_bf16,
                              const float* bias0, const uint16_t* W1, int N1, uint16_t* out1_bf16,
                              __half* out1_h, int8_t* out1_s, int actq1, const uint16_t* x, int T,
                              int K, uint32_t* err, cudaStream_t s, uint8_t* out1_q, uint8_t* out1_qs, int q1P,
                              float* out1_f32, const uint16_t* W0b, const uint16_t* xb, int Kb, int* zero,
                              int nzero) {
  if (T <= 0) return cudaSuccess;
  if (W0b && (W1 || !xb || Kb <= 0 || Kb % 64)) return cudaErrorInvalidValue;
  DenseArgs a{};
  a.p[0] = DenseProblem{N0, out0_f32, bias0, out0_bf16, nullptr, nullptr, 0, nullptr, nullptr, 0};
  a.p[1] = DenseProblem{N1, out1_f32, nullptr, out1_bf16, out1_h, out1_s, actq1, out1_q, out1_qs, q1P};
  if (out1_q && (!out1_bf16 || N1 % 32 != 0 || (q1P != 1 && q1P != 2))) return cudaErrorInvalidValue;
  a.units0 = W0 ? (N0 + kUnitRows - 1) / kUnitRows : 0;
  a.units = a.units0 + (W1 ? (N1 + kUnitRows - 1) / kUnitRows : 0);
  a.T = T;
  a.K = K;
  a.err = err;
  a.zero = zero;
  a.nzero = zero ? nzero : 0;
  if (a.units == 0) return cudaSuccess;
  const uint16_t* W[2] = {W0, W1};
  const int N[2] = {N0, N1};
  const int K2 = W0b ? Kb : 0;
  if (T <= 8) return launch_t<1>(a, W, N, x, W0b, xb, K2, s);
  if (T <= 16) return launch_t<2>(a, W, N, x, W0b, xb, K2, s);
  return launch_t<4>(a, W, N, x, W0b, xb, K2, s);  // chunks of 32 tokens
}

}  // namespace k3moe
