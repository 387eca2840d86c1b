// MXFP4 expert FFN for few rows per expert (decode): gate/up with the fused GLU, then down.
//
// "kimi-k3-in-c", MXFP4 experts: every weight is a 4-bit code indexing a 16-entry table and
// 32 consecutive weights share one 8-bit exponent; "kimi-k3-mlx", quantisation tiers: codes
// are packed low nibble first with e8m0 scales. For sorted row r of expert e (token t):
//   GLU pass:  a[r] = bf16(silu(G_e z_t) * (U_e z_t))          G_e, U_e [I][L]
//   down pass: o[r] = D_e a[r]                                  D_e [L][I]
//
// HBM-bound: only the selected experts' bytes are read, each once per chunk of up to 8 rows.
// A persistent CTA walks units = (chunk of rows of one expert, block of 32 output features).
// A producer warp streams the unit's code rows through a ring of shared-memory stages with
// per-row bulk copies (TMA engine) and its e8m0 scale rows into a double-buffered unit slot.
// Eight consumer warps split each stage's K. Per 32-weight block a warp converts the codes
// with the hardware e2m1 -> f16 conversion, multiplies them on the tensor cores (mma.sync
// m16n8k16, weights on M, rows on N) into a fresh fp32 block sum, and adds that sum scaled by
// 2^(E-127) (the e8m0 weight scale) times 2^s (the activation block scale). Activations arrive
// as an f16 copy with one power-of-two exponent per 32 values, so no value overflows f16 and
// every bf16 input from 2^-29 of its block maximum upwards converts exactly. A fixed-order
// shared-memory reduction over the warps keeps results deterministic.
//
// GLU unit: M-tile p holds gate rows 8p..8p+7 of the feature block as tile rows 0..7 and the
// matching up rows as tile rows 8..15, so one thread ends up with gate and up of a feature.
#include <cuda_fp16.h>

#include "k3moe_device.cuh"
#include "k3moe_internal.cuh"

namespace k3moe {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = 32 * (1 + kConsumerWarps);
constexpr int kStages = 6;

struct ExpertArgs {
  const uint8_t* q0;   // GLU: gate codes; down: down codes   [E][N][K/2]
  const uint8_t* s0;   //                                        [E][N][K/32]
  const uint8_t* q1;   // GLU: up codes (unused for down)
  const uint8_t* s1;
  int N, K;            // output features per expert, reduction length
  int KCB;             // code bytes per row per stage
  const int32_t* plan;
  const int32_t* offsets;
  const int32_t* row_token;  // GLU: B row = token of the sorted row; down: B row = sorted row
  const __half* bh;    // activations, f16 block-scaled [rows][K]
  const int8_t* bs;    // activation block exponents [rows][K/32]
  uint16_t* a_out;     // GLU output bf16 [rows][N]
  __half* ah_out;      // GLU output f16 block-scaled copy
  int8_t* as_out;
  float* o_out;        // down output fp32 [rows][N]
  int E;
  int actq;
  uint32_t* err;
};

struct Unit {
  int e, r0, nrows, fb;
};

__device__ __forceinline__ Unit decode_unit(const ExpertArgs& A, int u, int fbs) {
  const int* plan = A.plan;
  const int D = plan[0];
  const int* active = plan + 2;
  const int* cpre = plan + 2 + A.E;
  const int c = u / fbs;
  // binary search: largest d with cpre[d] <= c
  int lo = 0, hi = D - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cpre[mid] <= c) lo = mid; else hi = mid - 1;
  }
  Unit r;
  r.e = active[lo];
  const int q = c - cpre[lo];
  const int beg = A.offsets[r.e], end = A.offsets[r.e + 1];
  r.r0 = beg + q * kGemvTokens;
  r.nrows = min(kGemvTokens, end - r.r0);
  r.fb = u % fbs;
  return r;
}

template <bool GLU>
__global__ void __launch_bounds__(kThreads, 1) expert_gemv_kernel(const __grid_constant__ ExpertArgs A) {
  constexpr int kRows = GLU ? 2 * kUnitRows : kUnitRows;  // A rows per unit
  constexpr int kMT = GLU ? 4 : 2;                        // M-tiles per unit
  extern __shared__ __align__(128) uint8_t smem[];
  const int K = A.K, KCB = A.KCB;
  const int row_stride = KCB + 16;
  const int stage_bytes = kRows * row_stride;
  const int srow = K / 32;                    // scale bytes per row
  const int sbytes = kRows * srow;            // scale bytes per unit
  const int sslot = (sbytes + 127) & ~127;
  uint8_t* stages = smem;
  uint8_t* sbuf = smem + kStages * stage_bytes;
  float* red = reinterpret_cast<float*>(sbuf + 2 * sslot);
  uint64_t* full = reinterpret_cast<uint64_t*>(red + kConsumerWarps * kRows * kGemvTokens);
  uint64_t* empty = full + kStages;
  uint64_t* sfull = empty + kStages;
  uint64_t* sempty = sfull + 2;
  uint64_t* cbar = sempty + 2;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(cbar + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sfull[s], 1);
      mbar_init(&sempty[s], kConsumerWarps);
    }
    mbar_init(cbar, 32 * kConsumerWarps);
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  const int fbs = A.N / kUnitRows;
  const int units = A.plan[1] * fbs;
  const int ub = (int)(((long long)units * blockIdx.x) / gridDim.x);
  const int ue = (int)(((long long)units * (blockIdx.x + 1)) / gridDim.x);
  const int nkc = (K / 2) / KCB;
  const size_t qmat = (size_t)A.N * (K / 2);   // code bytes per expert matrix
  const size_t smat = (size_t)A.N * srow;      // scale bytes per expert matrix

  if (warp == 0) {
    // ---------------- producer
    int s = 0, us = 0;
    uint32_t ph = 0, uph = 0;
    bool ok = true;
    for (int u = ub; u < ue && ok; ++u) {
      const Unit U = decode_unit(A, u, fbs);
      const int f0 = U.fb * kUnitRows;
      if (!mbar_wait_bounded(&sempty[us], uph ^ 1, abort_flag, A.err)) { ok = false; break; }
      if (lane == 0) {
        mbar_arrive_expect_tx(&sfull[us], (uint32_t)sbytes);
        bulk_g2s(sbuf + us * sslot, A.s0 + U.e * smat + (size_t)f0 * srow, kUnitRows * srow, &sfull[us]);
        if (GLU)
          bulk_g2s(sbuf + us * sslot + kUnitRows * srow, A.s1 + U.e * smat + (size_t)f0 * srow,
                   kUnitRows * srow, &sfull[us]);
      }
      if (++us == 2) { us = 0; uph ^= 1; }
      for (int kc = 0; kc < nkc; ++kc) {
        if (!mbar_wait_bounded(&empty[s], ph ^ 1, abort_flag, A.err)) { ok = false; break; }
        if (lane == 0) mbar_arrive_expect_tx(&full[s], (uint32_t)(kRows * KCB));
        __syncwarp();
        uint8_t* dst = stages + s * stage_bytes;
        const size_t col = (size_t)kc * KCB;
        bulk_g2s(dst + lane * row_stride, A.q0 + U.e * qmat + (size_t)(f0 + lane) * (K / 2) + col, KCB,
                 &full[s]);
        if (GLU)
          bulk_g2s(dst + (kUnitRows + lane) * row_stride,
                   A.q1 + U.e * qmat + (size_t)(f0 + lane) * (K / 2) + col, KCB, &full[s]);
        if (++s == kStages) { s = 0; ph ^= 1; }
      }
    }
    if (!ok) {
      for (int i = 0; i < kStages; ++i) {
        if (--s < 0) { s = kStages - 1; ph ^= 1; }
        volatile int dummy = 0;
        mbar_wait_bounded(&full[s], ph, &dummy, A.err);
      }
    }
    return;
  }

  // ---------------- consumers
  const int cw = warp - 1;
  const int g = lane >> 2, t = lane & 3;
  const int kb_per_stage = KCB / 16;  // 32-weight blocks per stage
  const int kb_per_warp = (kb_per_stage + kConsumerWarps - 1) / kConsumerWarps;
  int s = 0, us = 0;
  uint32_t ph = 0, uph = 0, cph = 0;
  for (int u = ub; u < ue; ++u) {
    const Unit U = decode_unit(A, u, fbs);
    const int f0 = U.fb * kUnitRows;
    // B row of this lane's column (tile column g)
    const bool bvalid = g < U.nrows;
    const int brow = bvalid ? (GLU ? A.row_token[U.r0 + g] : U.r0 + g) : 0;
    const __half* bptr = A.bh + (size_t)brow * K;
    const int8_t* bsp = A.bs + (size_t)brow * (K / 32);

    float acc[kMT][4];
#pragma unroll
    for (int m = 0; m < kMT; ++m)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[m][i] = 0.f;

    if (!mbar_wait_bounded(&sfull[us], uph, abort_flag, A.err)) return;
    const uint8_t* sc = sbuf + us * sslot;

    for (int kc = 0; kc < nkc; ++kc) {
      if (!mbar_wait_bounded(&full[s], ph, abort_flag, A.err)) return;
      const uint8_t* sb = stages + s * stage_bytes;
      for (int i = 0; i < kb_per_warp; ++i) {
        const int kb = cw * kb_per_warp + i;
        if (kb >= kb_per_stage) break;
        const int KB = kc * kb_per_stage + kb;  // global 32-block index along K
        uint4 b = make_uint4(0, 0, 0, 0);
        int bexp = 0;
        if (bvalid) {
          b = ldg_nc_v4(bptr + KB * 32 + 8 * t);
          bexp = bsp[KB];
        }
        // activation block scale of tile columns 2t and 2t+1 (held by lanes 8t and 8t+4)
        const float sc0 = exp2i(__shfl_sync(0xffffffffu, bexp, 8 * t));
        const float sc1 = exp2i(__shfl_sync(0xffffffffu, bexp, 8 * t + 4));
#pragma unroll
        for (int m = 0; m < kMT; ++m) {
          // tile rows g and g+8 -> shared-memory rows
          const int rlo = GLU ? (8 * m + g) : (16 * m + g);
          const int rhi = GLU ? (kUnitRows + 8 * m + g) : (16 * m + g + 8);
          const uint32_t qlo = *reinterpret_cast<const uint32_t*>(sb + rlo * row_stride + kb * 16 + 4 * t);
          const uint32_t qhi = *reinterpret_cast<const uint32_t*>(sb + rhi * row_stride + kb * 16 + 4 * t);
          const float slo = e8m0_to_f32(sc[rlo * srow + KB]);
          const float shi = e8m0_to_f32(sc[rhi * srow + KB]);
          float tmp[4] = {0.f, 0.f, 0.f, 0.f};
          mma_f16(tmp, e2m1x2_to_f16x2(qlo & 0xff), e2m1x2_to_f16x2(qhi & 0xff),
                  e2m1x2_to_f16x2((qlo >> 8) & 0xff), e2m1x2_to_f16x2((qhi >> 8) & 0xff), b.x, b.y);
          mma_f16(tmp, e2m1x2_to_f16x2((qlo >> 16) & 0xff), e2m1x2_to_f16x2((qhi >> 16) & 0xff),
                  e2m1x2_to_f16x2(qlo >> 24), e2m1x2_to_f16x2(qhi >> 24), b.z, b.w);
          acc[m][0] = fmaf(tmp[0], slo * sc0, acc[m][0]);
          acc[m][1] = fmaf(tmp[1], slo * sc1, acc[m][1]);
          acc[m][2] = fmaf(tmp[2], shi * sc0, acc[m][2]);
          acc[m][3] = fmaf(tmp[3], shi * sc1, acc[m][3]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      if (++s == kStages) { s = 0; ph ^= 1; }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sempty[us]);
    if (++us == 2) { us = 0; uph ^= 1; }

    // fixed-order reduction over the consumer warps; red[w][row][col]
    float* r = red + cw * kRows * kGemvTokens;
#pragma unroll
    for (int m = 0; m < kMT; ++m) {
      const int rlo = GLU ? (8 * m + g) : (16 * m + g);
      const int rhi = GLU ? (kUnitRows + 8 * m + g) : (16 * m + g + 8);
      r[rlo * kGemvTokens + 2 * t] = acc[m][0];
      r[rlo * kGemvTokens + 2 * t + 1] = acc[m][1];
      r[rhi * kGemvTokens + 2 * t] = acc[m][2];
      r[rhi * kGemvTokens + 2 * t + 1] = acc[m][3];
    }
    if (!group_barrier(cbar, cph, abort_flag, A.err)) return;
    // epilogue: warp cw handles column (row of the chunk) cw, lane = feature f0 + lane
    if (cw < U.nrows) {
      const int row = U.r0 + cw;
      if (GLU) {
        float gs = 0.f, us_ = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
          gs += red[(w * kRows + lane) * kGemvTokens + cw];
          us_ += red[(w * kRows + kUnitRows + lane) * kGemvTokens + cw];
        }
        const float av = gs / (1.0f + expf(-gs)) * us_;
        const uint16_t ab = f32_to_bf16(av);
        A.a_out[(size_t)row * A.N + f0 + lane] = ab;
        float q = bf16_to_f32(ab);
        if (A.actq) q = mxfp8_roundtrip(q, mxfp8_block_exp(warp_max(fabsf(q))));
        const int e = f16_block_exp(warp_max(fabsf(q)));
        A.ah_out[(size_t)row * A.N + f0 + lane] = __float2half_rn(ldexpf(q, -e));
        if (lane == 0) A.as_out[(size_t)row * (A.N / 32) + U.fb] = (int8_t)e;
      } else {
        float o = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) o += red[(w * kRows + lane) * kGemvTokens + cw];
        A.o_out[(size_t)row * A.N + f0 + lane] = o;
      }
    }
    if (!group_barrier(cbar, cph, abort_flag, A.err)) return;
  }
}

template <bool GLU>
cudaError_t launch_t(const ExpertArgs& a, int units_max, cudaStream_t s) {
  constexpr int kRows = GLU ? 2 * kUnitRows : kUnitRows;
  const int row_stride = a.KCB + 16;
  const int sbytes = kRows * (a.K / 32);
  const int sslot = (sbytes + 127) & ~127;
  const size_t smem = (size_t)kStages * kRows * row_stride + 2 * (size_t)sslot +
                      (size_t)kConsumerWarps * kRows * kGemvTokens * sizeof(float) +
                      (2 * kStages + 5) * sizeof(uint64_t) + 16;
  cudaError_t e = cudaFuncSetAttribute(expert_gemv_kernel<GLU>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int grid = num_sms();
  if (units_max < grid) grid = units_max > 0 ? units_max : 1;
  expert_gemv_kernel<GLU><<<grid, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

int pick_kcb(int row_bytes) {
  for (int c : {256, 128, 64, 32, 16})
    if (row_bytes % c == 0) return c;
  return 16;
}

}  // namespace

cudaError_t launch_expert_glu(const k3moe_dims& d, const k3moe_weights& w, const int32_t* plan,
                              const int32_t* offsets, const int32_t* row_token, const __half* zh,
                              const int8_t* zs, uint16_t* a, __half* ah, int8_t* as, int rows_max,
                              uint32_t* err, cudaStream_t s) {
  ExpertArgs A{};
  A.q0 = w.gate_q; A.s0 = w.gate_s; A.q1 = w.up_q; A.s1 = w.up_s;
  A.N = d.inter; A.K = d.latent; A.KCB = pick_kcb(d.latent / 2);
  A.plan = plan; A.offsets = offsets; A.row_token = row_token;
  A.bh = zh; A.bs = zs; A.a_out = a; A.ah_out = ah; A.as_out = as;
  A.E = d.n_experts; A.actq = d.actq; A.err = err;
  const int chunks_max = rows_max / kGemvTokens + d.n_experts;
  return launch_t<true>(A, chunks_max * (d.inter / kUnitRows), s);
}

cudaError_t launch_expert_down(const k3moe_dims& d, const k3moe_weights& w, const int32_t* plan,
                               const int32_t* offsets, const __half* ah, const int8_t* as,
                               float* o_rows, int rows_max, uint32_t* err, cudaStream_t s) {
  ExpertArgs A{};
  A.q0 = w.down_q; A.s0 = w.down_s;
  A.N = d.latent; A.K = d.inter; A.KCB = pick_kcb(d.inter / 2);
  A.plan = plan; A.offsets = offsets; A.row_token = nullptr;
  A.bh = ah; A.bs = as; A.o_out = o_rows;
  A.E = d.n_experts; A.actq = d.actq; A.err = err;
  const int chunks_max = rows_max / kGemvTokens + d.n_experts;
  return launch_t<false>(A, chunks_max * (d.latent / kUnitRows), s);
}

}  // namespace k3moe
