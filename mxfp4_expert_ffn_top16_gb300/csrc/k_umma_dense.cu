// Dense bf16 projections for many tokens (prefill) on the 5th-generation tensor cores:
// router logits, latent in, latent out ("kimi-k3-mlx", Architecture table: router over 896
// experts; Stable LatentMoE: 7168 -> 3584 -> 7168 around the routed experts).
//
//   out[t][n] = sum_k W[n][k] x[t][k]
//
// A persistent CTA walks 128 x BN output tiles (128 weight rows on M, BN tokens on N; BN = 256
// for many tokens: 48 KB of operands per 4.2 MFLOP stage, twice the flops per byte from L2 of
// BN = 64, which is kept for a few hundred tokens, where 256-token tiles would leave SMs idle).
// Warp 0 streams 128 x 64 bf16 tiles of W and BN x 64 tiles of x through TMA (128-byte
// swizzle) into a ring of stages. Warp 1 allocates the tensor memory (BN-column accumulator
// slots) and issues tcgen05.mma kind::f16 (M=128, N=BN, K=16, four per stage); each group of 4
// stages (256 of K) accumulates into one slot, which is committed to the epilogue. The
// epilogue warps (lane quadrant = warp % 4; with BN = 256 two warps per quadrant, half of the
// columns each; one tensor-memory lane = one weight row per thread) drain every slot into
// per-thread fp32 sums added in group order, so the tensor core's own accumulation spans at
// most 16 MMAs. (Each MMA rounds its running sum once: with 16-MMA groups the fp32 logits of
// K = 7168 are within 3.2e-7 of their exact values on average, half the error of 32-MMA groups,
// for ~6% more time in this kernel; the bf16 roundings of z then follow the exact sums as often
// as a plain fp32 evaluation on the CPU does.) After the last group they write fp32 + bias
// (logits), bf16 (z, y) and, for z,
// the f16 block-scaled copy with one power-of-two exponent per 32 features (in MXFP8 mode of
// the MXFP8 round trip).
#include <cuda_fp16.h>

#include "k3moe_device.cuh"
#include "k3moe_internal.cuh"
#include "k3moe_umma.cuh"

namespace k3moe {
namespace {

constexpr int BM = 128, BK = 64, kGroup = 4, kGroupM = 16;
constexpr int kATile = BM * BK * 2;  // 16 KB
template <int BN>
struct Tile {
  static constexpr int kStages = BN == 256 ? 4 : 6;
  static constexpr int kSlots = BN == 256 ? 2 : 4;
  static constexpr int kBTile = BN * BK * 2;
  static constexpr int kEpiWarps = BN == 256 ? 8 : 4;
  static constexpr int kThreads = 32 * (2 + kEpiWarps);
  static constexpr int kEpiCols = BN / (kEpiWarps / 4);  // accumulator columns (tokens) per epilogue warp
  static constexpr uint32_t kTmemCols = kSlots * BN;
  static_assert(kTmemCols <= 512 && (kTmemCols & (kTmemCols - 1)) == 0, "tensor memory");
  static constexpr size_t kSmem = 1024 + (size_t)kStages * (kATile + kBTile) + (2 * kStages + 2 * kSlots + 1) * 8 + 16;
  static_assert(kSmem <= 227 * 1024, "shared memory");
};

struct UProblem {
  int N;
  float* out_f32;
  const float* bias;
  uint16_t* out_bf16;
  __half* out_h;
  int8_t* out_s;
  int actq;
};

struct UDenseArgs {
  CUtensorMap tw[2];  // W of each problem: {K, N} bf16, box {64, 128}, 128-byte swizzle
  CUtensorMap tx;     // tokens: {K, T} bf16, box {64, 64}, 128-byte swizzle
  UProblem p[2];
  int mt0, mtiles, ntiles;
  int T, K;
  // optional second K segment of problem 0 (a single problem): out = W x + W2 x2, W2 {K2, N0},
  // x2 {K2, T}; its K steps follow the first nk0
  CUtensorMap tw2, tx2;
  int nk0, K2;
  uint32_t* err;
};

template <int BN>
__global__ void __launch_bounds__(Tile<BN>::kThreads, 1) umma_dense_kernel(const __grid_constant__ UDenseArgs a) {
  using TL = Tile<BN>;
  constexpr int kStages = TL::kStages, kSlots = TL::kSlots, kBTile = TL::kBTile, kEpiWarps = TL::kEpiWarps,
                kEpiCols = TL::kEpiCols;
  constexpr uint32_t kTmemCols = TL::kTmemCols;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kATile;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + kStages * kBTile);
  uint64_t* empty = full + kStages;
  uint64_t* accf = empty + kStages;
  uint64_t* acce = accf + kSlots;
  uint64_t* drain = acce + kSlots;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < kSlots; ++b) {
      mbar_init(&accf[b], 1);
      mbar_init(&acce[b], kEpiWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_wait();
  pdl_trigger();
  const uint32_t tmem = *tmem_slot;
  const int items = a.mtiles * a.ntiles;
  const int nk = a.K / BK + a.K2 / BK;
  // item -> (weight tile, token tile), in groups of kGroupM weight tiles: the CTAs in flight
  // share a few weight tiles and a few token tiles, so both are reused from L2 even when the
  // tokens do not fit in it
  auto tile_of = [&](int it, int& mt, int& nt) {
    const int g = it / (kGroupM * a.ntiles), r = it - g * kGroupM * a.ntiles;
    const int gm = min(kGroupM, a.mtiles - g * kGroupM);
    nt = r / gm;
    mt = g * kGroupM + (r - nt * gm);
  };
  const int ngroups = (nk + kGroup - 1) / kGroup;

  if (warp == 0) {
    if (lane == 0) {  // ---------------- TMA producer
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
        int mt, nt;
        tile_of(it, mt, nt);
        const int pi = mt < a.mt0 ? 0 : 1;
        const int row0 = (pi ? mt - a.mt0 : mt) * BM;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait_bounded(&empty[s], ph ^ 1, abort_flag, a.err)) { ok = false; break; }
          mbar_arrive_expect_tx(&full[s], kATile + kBTile);
          if (kb < a.nk0) {
            tma_load_2d(sA + s * kATile, &a.tw[pi], kb * BK, row0, &full[s]);
            tma_load_2d(sB + s * kBTile, &a.tx, kb * BK, nt * BN, &full[s]);
          } else {  // second K segment (problem 0 only)
            tma_load_2d(sA + s * kATile, &a.tw2, (kb - a.nk0) * BK, row0, &full[s]);
            tma_load_2d(sB + s * kBTile, &a.tx2, (kb - a.nk0) * BK, nt * BN, &full[s]);
          }
          if (++s == kStages) { s = 0; ph ^= 1; }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ---------------- MMA issuer
      constexpr uint32_t idesc = idesc_bf16(BM, BN);
      int s = 0, slot = 0;
      uint32_t ph = 0, sph = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
        for (int gi = 0; gi < ngroups && ok; ++gi) {
          if (!mbar_wait_bounded(&acce[slot], sph ^ 1, abort_flag, a.err)) { ok = false; break; }
          tc_fence_after();
          const uint32_t d = tmem + (uint32_t)(slot * BN);
          const int kb1 = min(nk, (gi + 1) * kGroup);
          for (int kb = gi * kGroup; kb < kb1; ++kb) {
            if (!mbar_wait_bounded(&full[s], ph, abort_flag, a.err)) { ok = false; break; }
            tc_fence_after();
            const uint32_t a0 = smem_u32(sA + s * kATile), b0 = smem_u32(sB + s * kBTile);
#pragma unroll
            for (int k = 0; k < BK / 16; ++k)
              umma_bf16(d, sdesc_sw128(a0 + k * 32), sdesc_sw128(b0 + k * 32), idesc,
                        (kb != gi * kGroup || k != 0) ? 1u : 0u);
            umma_commit(&empty[s]);
            if (++s == kStages) { s = 0; ph ^= 1; }
          }
          if (!ok) break;
          umma_commit(&accf[slot]);
          if (++slot == kSlots) { slot = 0; sph ^= 1; }
        }
      }
      // every issued MMA has completed before the tensor memory is released
      umma_commit(drain);
      volatile int no_abort = 0;
      mbar_wait_bounded(drain, 0, &no_abort, a.err);
    }
  } else {  // ---------------- epilogue warps 2..9: lane quadrant = warp % 4, column half h
    const int q = warp & 3, h = (warp - 2) >> 2;
    int slot = 0;
    uint32_t sph = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
      int mt, nt;
      tile_of(it, mt, nt);
      const int pi = mt < a.mt0 ? 0 : 1;
      const UProblem& P = a.p[pi];
      const int row = (pi ? mt - a.mt0 : mt) * BM + q * 32 + lane;  // output feature
      float sum[kEpiCols];
#pragma unroll
      for (int j = 0; j < kEpiCols; ++j) sum[j] = 0.f;
      for (int gi = 0; gi < ngroups; ++gi) {
        if (!mbar_wait_warp(&accf[slot], sph, abort_flag, a.err)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < kEpiCols; c += 32) {
          uint32_t v[32];
          tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(slot * BN + h * kEpiCols + c), v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) sum[c + j] += __uint_as_float(v[j]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acce[slot]);
        if (++slot == kSlots) { slot = 0; sph ^= 1; }
      }
      if (!ok) break;
      const bool valid = row < P.N;
      // outputs of this warp: tokens tok0 .. tok0 + ntok - 1, one loop per output kind (the
      // executed code per item stays small: the MMA and TMA warps' loops stay in the
      // instruction cache)
      const int tok0 = nt * BN + h * kEpiCols;
      const int ntok = min(kEpiCols, a.T - tok0);
      if (P.out_h) {  // f16 block-scaled copy (+ bf16): N multiple of 32, the warp's rows are one block
#pragma unroll
        for (int j = 0; j < kEpiCols; ++j) {
          if (j >= ntok) continue;  // uniform across the warp
          const int tok = tok0 + j;
          const uint16_t vb = f32_to_bf16(sum[j]);
          if (valid) P.out_bf16[(size_t)tok * P.N + row] = vb;
          float qv = bf16_to_f32(vb);
          if (P.actq) qv = mxfp8_roundtrip(qv, mxfp8_block_exp(warp_max(fabsf(qv))));
          const int e = f16_block_exp(warp_max(fabsf(qv)));
          if (valid) {
            P.out_h[(size_t)tok * P.N + row] = __float2half_rn(ldexpf(qv, -e));
            if (lane == 0) P.out_s[(size_t)tok * exp_pitch(P.N) + row / 32] = (int8_t)e;
          }
        }
      } else if (valid && P.out_f32) {  // router logits + bias
        const float bias = P.bias ? P.bias[row] : 0.f;
        float* dst = P.out_f32 + (size_t)tok0 * P.N + row;
#pragma unroll
        for (int j = 0; j < kEpiCols; ++j) {
          if (j < ntok) *dst = sum[j] + bias;
          dst += P.N;
        }
      } else if (valid && P.out_bf16) {
        uint16_t* dst = P.out_bf16 + (size_t)tok0 * P.N + row;
#pragma unroll
        for (int j = 0; j < kEpiCols; ++j) {
          if (j < ntok) *dst = f32_to_bf16(sum[j]);
          dst += P.N;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int BN>
cudaError_t launch_bn(UDenseArgs& a, const uint16_t* const W[2], const int N[2], const uint16_t* x, int T, int K,
                      const uint16_t* W2, const uint16_t* x2, cudaStream_t s) {
  a.ntiles = (T + BN - 1) / BN;
  for (int i = 0; i < 2; ++i)
    if (W[i] && !make_tmap_2d(&a.tw[i], W[i], 2, (uint64_t)K, (uint64_t)N[i], (uint64_t)K * 2, BK, BM, true))
      return cudaErrorInvalidValue;
  if (!make_tmap_2d(&a.tx, x, 2, (uint64_t)K, (uint64_t)T, (uint64_t)K * 2, BK, BN, true))
    return cudaErrorInvalidValue;
  if (a.K2 > 0 && (!make_tmap_2d(&a.tw2, W2, 2, (uint64_t)a.K2, (uint64_t)N[0], (uint64_t)a.K2 * 2, BK, BM, true) ||
                   !make_tmap_2d(&a.tx2, x2, 2, (uint64_t)a.K2, (uint64_t)T, (uint64_t)a.K2 * 2, BK, BN, true)))
    return cudaErrorInvalidValue;
  constexpr size_t smem = Tile<BN>::kSmem;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(umma_dense_kernel<BN>), smem);
  if (e != cudaSuccess) return e;
  const int items = a.mtiles * a.ntiles;
  const int grid = items < num_sms() ? items : num_sms();
  return launch_pdl(umma_dense_kernel<BN>, dim3(grid), dim3(Tile<BN>::kThreads), smem, s, a);
}

}  // namespace

cudaError_t launch_umma_dense(const uint16_t* W0, int N0, float* out0_f32, uint16_t* out0_bf16,
                              const float* bias0, const uint16_t* W1, int N1, uint16_t* out1_bf16,
                              __half* out1_h, int8_t* out1_s, int actq1, const uint16_t* x, int T, int K,
                              uint32_t* err, cudaStream_t s, float* out1_f32, const uint16_t* W0b,
                              const uint16_t* xb, int Kb) {
  if (T <= 0) return cudaSuccess;
  // one output kind per problem: fp32 (+ bias), bf16, or bf16 + the f16 block-scaled copy
  if ((out0_f32 && out0_bf16) || (out1_f32 && (out1_bf16 || out1_h))) return cudaErrorInvalidValue;
  if (W0b && (W1 || !xb || Kb <= 0 || Kb % BK)) return cudaErrorInvalidValue;
  UDenseArgs a{};
  a.p[0] = UProblem{N0, out0_f32, bias0, out0_bf16, nullptr, nullptr, 0};
  a.p[1] = UProblem{N1, out1_f32, nullptr, out1_bf16, out1_h, out1_s, actq1};
  a.nk0 = K / BK;
  a.K2 = W0b ? Kb : 0;
  a.mt0 = W0 ? (N0 + BM - 1) / BM : 0;
  a.mtiles = a.mt0 + (W1 ? (N1 + BM - 1) / BM : 0);
  a.T = T;
  a.K = K;
  a.err = err;
  const uint16_t* W[2] = {W0, W1};
  const int N[2] = {N0, N1};
  // rounds of items over the SMs times the cost of one item (a 256-token tile ~ two 64-token ones)
  const long long g = num_sms();
  const long long r64 = ((long long)a.mtiles * ((T + 63) / 64) + g - 1) / g;
  const long long r256 = ((long long)a.mtiles * ((T + 255) / 256) + g - 1) / g;
  if (2 * r256 < r64) return launch_bn<256>(a, W, N, x, T, K, W0b, xb, s);
  return launch_bn<64>(a, W, N, x, T, K, W0b, xb, s);
}

}  // namespace k3moe
