// MXFP4 expert FFN for few rows per expert (decode): gate/up with the fused GLU, then down.
//
// "kimi-k3-in-c", MXFP4 experts: every weight is a 4-bit code indexing a 16-entry table and
// 32 consecutive weights share one 8-bit exponent; "kimi-k3-mlx", quantisation tiers: codes
// are packed low nibble first with e8m0 scales. For sorted row r of expert e (token t):
//   GLU pass:  a[r] = bf16(silu(G_e z_t) * (U_e z_t))          G_e, U_e [I][L]
//   down pass: o[r] = D_e a[r]                                  D_e [L][I]
//
// HBM-bound: only the selected experts' bytes are read, each once per chunk of up to 8 rows.
// A persistent CTA walks a contiguous range of units = (chunk of rows of one expert, block of
// 32 output features); the chunk table gives a unit's expert and rows in one load. A producer
// warp streams, through the TMA engine:
//   - code tiles of 32 rows x 128 bytes (256 weights, 128-byte swizzle), two per stage
//     (GLU: gate and up at the same K; down: two consecutive K ranges), into a deep ring of
//     shared-memory stages,
//   - the unit's e8m0 scale rows (one contiguous 1-D copy per matrix) into a double-buffered
//     unit slot,
//   - the chunk's activation rows (f16, block-scaled) and block exponents into an activation
//     slot, reloaded only when the chunk changes.
// Few large copies matter: the TMA engine takes roughly one copy per ~60 cycles per SM, so
// per-row copies of a few hundred bytes cannot reach HBM bandwidth while 4-8 KB tiles can.
// Sixteen consumer warps share each stage: warp w takes 32-weight block (w mod 8) of a tile
// and, for the GLU, half of the unit's M-tiles (for down, one of the two tiles). Per block a
// warp converts the codes with the hardware e2m1 -> f16 conversion, multiplies them on the
// tensor cores (mma.sync m16n8k16, weights on M, rows on N) into a fresh fp32 block sum, and
// adds that sum times 2^(E-127) (the e8m0 weight scale) times 2^s (the activation block
// scale). Activations are an f16 copy with one power-of-two exponent per 32 values, so no
// value overflows f16 and every bf16 input from 2^-29 of its block maximum upwards converts
// exactly. A fixed-order shared-memory reduction over the warps keeps results deterministic.
//
// GLU unit: M-tile p holds gate rows 8p..8p+7 of the feature block as tile rows 0..7 and the
// matching up rows as tile rows 8..15, so one thread ends up with gate and up of a feature.
//
// Inputs are checked on the device: a chunk whose expert is out of range or a row token
// outside [0, T) sets the index bit of the error word and the affected rows are skipped.
#include <cuda_fp16.h>

#include "k3moe_device.cuh"
#include "k3moe_internal.cuh"

namespace k3moe {
namespace {

constexpr int kConsumerWarps = 16;
constexpr int kThreads = 32 * (1 + kConsumerWarps);
constexpr int kMaxStages = 24;
constexpr int kStageBudget = 96 * 1024;
constexpr int kTileRows = kUnitRows;  // rows per code tile

struct ExpertArgs {
  CUtensorMap tq0;     // GLU: gate codes; down: down codes. 2-D {K/2 bytes, E*N rows}
  CUtensorMap tq1;     // GLU: up codes
  const uint8_t* s0;   // scales [E][N][K/32]
  const uint8_t* s1;   // GLU: up scales
  int N, K;            // output features per expert, reduction length
  int IB;              // code bytes per tile row (128, or 64/32 for small K)
  int NS;              // ring stages
  const int32_t* plan;
  const int4* ctab;
  const int32_t* row_token;  // GLU: B row = token of the sorted row; down: B row = sorted row
  int brows;           // rows of the activation arrays (GLU: T, down: T*k)
  int rows_max;        // T*k
  const __half* bh;    // activations, f16 block-scaled [brows][K]
  const int8_t* bs;    // activation block exponents [brows][exp_pitch(K)]
  uint16_t* a_out;     // GLU output bf16 [rows][N]
  __half* ah_out;      // GLU output f16 block-scaled copy [rows][N]
  int8_t* as_out;      // its exponents [rows][exp_pitch(N)]
  float* o_out;        // down output fp32 [rows][N]
  int E;
  int actq;
  uint32_t* err;
};

struct Unit {
  int e, r0, nrows, fb, chunk;
};

__device__ __forceinline__ Unit decode_unit(const ExpertArgs& A, int u, int fbs, bool report) {
  Unit r;
  r.chunk = u / fbs;
  r.fb = u - r.chunk * fbs;
  const int4 c = A.ctab[r.chunk];
  const bool ok = c.x >= 0 && c.x < A.E && c.y >= 0 && c.z >= 0 && c.z <= kGemvTokens &&
                  c.y + c.z <= A.rows_max;
  r.e = ok ? c.x : 0;
  r.r0 = ok ? c.y : 0;
  r.nrows = ok ? c.z : 0;
  if (!ok && report) atomicOr(A.err, kErrIndex);
  return r;
}

// One 32-weight block for two M-tiles: codes at byte offsets q0/q1 (tile rows g, g+8 of
// M-tile 0) and q2/q3 (M-tile 1), e8m0 scales s0..s3 of those rows, activation fragment b and
// the activation scales of tile columns 2t, 2t+1.
__device__ __forceinline__ void block_mma(float (&acc)[2][4], const uint8_t* sb, int q0, int q1, int q2,
                                          int q3, float s0, float s1, float s2, float s3, uint4 b,
                                          float sc0, float sc1) {
  const uint32_t w[4] = {*reinterpret_cast<const uint32_t*>(sb + q0), *reinterpret_cast<const uint32_t*>(sb + q1),
                         *reinterpret_cast<const uint32_t*>(sb + q2), *reinterpret_cast<const uint32_t*>(sb + q3)};
  const float sl[4] = {s0, s1, s2, s3};
#pragma unroll
  for (int m = 0; m < 2; ++m) {
    uint32_t lo[4], hi[4];
    e2m1x8_to_f16x2x4(w[2 * m], lo);
    e2m1x8_to_f16x2x4(w[2 * m + 1], hi);
    float tmp[4] = {0.f, 0.f, 0.f, 0.f};
    mma_f16(tmp, lo[0], hi[0], lo[1], hi[1], b.x, b.y);
    mma_f16(tmp, lo[2], hi[2], lo[3], hi[3], b.z, b.w);
    acc[m][0] = fmaf(tmp[0], sl[2 * m] * sc0, acc[m][0]);
    acc[m][1] = fmaf(tmp[1], sl[2 * m] * sc1, acc[m][1]);
    acc[m][2] = fmaf(tmp[2], sl[2 * m + 1] * sc0, acc[m][2]);
    acc[m][3] = fmaf(tmp[3], sl[2 * m + 1] * sc1, acc[m][3]);
  }
}

template <bool GLU>
__global__ void __launch_bounds__(kThreads, 1) expert_gemv_kernel(const __grid_constant__ ExpertArgs A) {
  constexpr int kRows = GLU ? 2 * kUnitRows : kUnitRows;  // weight rows per unit
  constexpr int kParts = GLU ? 8 : 16;                    // partial sums per output row
  extern __shared__ __align__(1024) uint8_t smem[];
  const int K = A.K, IB = A.IB, NS = A.NS;
  const int tile_bytes = kTileRows * IB;
  const int stage_bytes = (2 * tile_bytes + 1023) & ~1023;
  const int ntiles = (K / 2) / IB;                         // tiles per weight row range
  const int nkc = GLU ? ntiles : (ntiles + 1) / 2;         // stages per unit
  const int srow = K / 32;                                 // scale bytes per weight row
  const int sbytes = kRows * srow;                         // scale bytes per unit
  const int sslot = (sbytes + 127) & ~127;
  const int bpitch = K * 2 + 64;                           // f16 activation row pitch in smem
  const int epitch = exp_pitch(K);                         // exponent row pitch
  const int bslot = kGemvTokens * bpitch + kGemvTokens * epitch;
  // stages start on a 1024-byte boundary of the shared window (the 128-byte swizzle pattern
  // is a function of the shared address)
  uint8_t* stages = smem + ((1024u - (smem_u32(smem) & 1023u)) & 1023u);
  uint8_t* sbuf = stages + NS * stage_bytes;
  uint8_t* bbuf = sbuf + 2 * sslot;
  const int8_t* bexp = reinterpret_cast<const int8_t*>(bbuf + kGemvTokens * bpitch);
  float* red = reinterpret_cast<float*>(bbuf + ((bslot + 127) & ~127));
  int* bidx = reinterpret_cast<int*>(red + kParts * kRows * kGemvTokens);
  uint64_t* full = reinterpret_cast<uint64_t*>(bidx + kGemvTokens);
  uint64_t* empty = full + kMaxStages;
  uint64_t* sfull = empty + kMaxStages;
  uint64_t* sempty = sfull + 2;
  uint64_t* bfull = sempty + 2;
  uint64_t* bempty = bfull + 1;
  uint64_t* cbar = bempty + 1;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(cbar + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sfull[s], 1);
      mbar_init(&sempty[s], kConsumerWarps);
    }
    mbar_init(bfull, 1);
    mbar_init(bempty, kConsumerWarps);
    mbar_init(cbar, kConsumerWarps);
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();

  const int fbs = A.N / kUnitRows;
  const int C = A.plan[1];
  const int units = (C > 0 && C <= A.rows_max / kGemvTokens + A.E) ? C * fbs : 0;
  const int ub = (int)(((long long)units * blockIdx.x) / gridDim.x);
  const int ue = (int)(((long long)units * (blockIdx.x + 1)) / gridDim.x);
  const size_t smat = (size_t)A.N * srow;  // scale bytes per expert matrix

  if (warp == 0) {
    // ---------------- producer (lane 0 issues; the warp stays converged)
    int s = 0, us = 0, cur = -1;
    uint32_t ph = 0, uph = 0, bph = 0;
    bool ok = true;
    for (int u = ub; u < ue && ok; ++u) {
      const Unit U = decode_unit(A, u, fbs, lane == 0);
      const int f0 = U.fb * kUnitRows;
      if (U.chunk != cur) {  // activation rows of a new chunk
        if (!mbar_wait_bounded(bempty, bph ^ 1, abort_flag, A.err)) { ok = false; break; }
        int br = -1;
        if (lane < U.nrows) {
          const int r = U.r0 + lane;
          br = GLU ? A.row_token[r] : r;
          if (br < 0 || br >= A.brows) {
            atomicOr(A.err, kErrIndex);
            br = -1;
          }
        }
        if (lane < kGemvTokens) bidx[lane] = br;
        const unsigned have = __ballot_sync(0xffffffffu, br >= 0);
        if (lane == 0) mbar_arrive_expect_tx(bfull, (uint32_t)(__popc(have) * (K * 2 + epitch)));
        __syncwarp();
        if (br >= 0) {
          bulk_g2s(bbuf + lane * bpitch, A.bh + (size_t)br * K, K * 2, bfull);
          bulk_g2s(bbuf + kGemvTokens * bpitch + lane * epitch, A.bs + (size_t)br * epitch, epitch, bfull);
        }
        bph ^= 1;
        cur = U.chunk;
      }
      if (!mbar_wait_bounded(&sempty[us], uph ^ 1, abort_flag, A.err)) { ok = false; break; }
      if (lane == 0) {
        mbar_arrive_expect_tx(&sfull[us], (uint32_t)sbytes);
        bulk_g2s(sbuf + us * sslot, A.s0 + U.e * smat + (size_t)f0 * srow, kUnitRows * srow, &sfull[us]);
        if (GLU)
          bulk_g2s(sbuf + us * sslot + kUnitRows * srow, A.s1 + U.e * smat + (size_t)f0 * srow,
                   kUnitRows * srow, &sfull[us]);
      }
      if (++us == 2) { us = 0; uph ^= 1; }
      const int y = U.e * A.N + f0;
      for (int kc = 0; kc < nkc; ++kc) {
        if (!mbar_wait_bounded(&empty[s], ph ^ 1, abort_flag, A.err)) { ok = false; break; }
        if (lane == 0) {
          uint8_t* dst = stages + s * stage_bytes;
          if (GLU) {
            mbar_arrive_expect_tx(&full[s], (uint32_t)(2 * tile_bytes));
            tma_load_2d(dst, &A.tq0, kc * IB, y, &full[s]);
            tma_load_2d(dst + tile_bytes, &A.tq1, kc * IB, y, &full[s]);
          } else {
            const int nt = (2 * kc + 1 < ntiles) ? 2 : 1;
            mbar_arrive_expect_tx(&full[s], (uint32_t)(nt * tile_bytes));
            tma_load_2d(dst, &A.tq0, 2 * kc * IB, y, &full[s]);
            if (nt == 2) tma_load_2d(dst + tile_bytes, &A.tq0, (2 * kc + 1) * IB, y, &full[s]);
          }
        }
        __syncwarp();
        if (++s == NS) { s = 0; ph ^= 1; }
      }
    }
    if (!ok) {
      for (int i = 0; i < NS; ++i) {
        if (--s < 0) { s = NS - 1; ph ^= 1; }
        volatile int dummy = 0;
        mbar_wait_bounded(&full[s], ph, &dummy, A.err);
      }
    }
    return;
  }

  // ---------------- consumers
  const int cw = warp - 1;
  const int g = lane >> 2, t = lane & 3;
  const int kb = cw & 7;          // 32-weight block inside a tile
  const int sel = cw >> 3;        // GLU: M-tile pair; down: tile of the stage
  const bool kb_on = kb < IB / 16;
  // byte offset of this lane's 4 code bytes in tile row g of a 128-byte-row tile (swizzled) or
  // of a narrower unswizzled tile; rows 8j + g share it up to j * 8 * IB
  const int lane_off = (IB == 128) ? g * 128 + ((kb ^ g) << 4) + 4 * t : g * IB + kb * 16 + 4 * t;
  // tile rows of this warp's two M-tiles (tile rows g and g+8 of each) -> shared-memory rows
  //   GLU:  M-tile p = 2*sel + m: gate row 8p + g (tile 0), up row 8p + g (tile 1)
  //   down: M-tile m: rows 16m + g and 16m + g + 8 of tile `sel`
  int q[4], srows[4];
#pragma unroll
  for (int m = 0; m < 2; ++m) {
    if (GLU) {
      const int p = 2 * sel + m;
      q[2 * m] = 8 * p * IB + lane_off;
      q[2 * m + 1] = tile_bytes + 8 * p * IB + lane_off;
      srows[2 * m] = 8 * p + g;
      srows[2 * m + 1] = kUnitRows + 8 * p + g;
    } else {
      q[2 * m] = sel * tile_bytes + 16 * m * IB + lane_off;
      q[2 * m + 1] = sel * tile_bytes + (16 * m + 8) * IB + lane_off;
      srows[2 * m] = 16 * m + g;
      srows[2 * m + 1] = 16 * m + g + 8;
    }
  }
  int s = 0, us = 0, cur = -1;
  uint32_t ph = 0, uph = 0, bph = 0, cph = 0;
  bool bvalid = false, v0 = false, v1 = false;
  for (int u = ub; u < ue; ++u) {
    const Unit U = decode_unit(A, u, fbs, false);
    const int f0 = U.fb * kUnitRows;
    if (U.chunk != cur) {
      if (cur != -1) {
        __syncwarp();
        if (lane == 0) mbar_arrive(bempty);
      }
      if (!mbar_wait_bounded(bfull, bph, abort_flag, A.err)) return;
      bph ^= 1;
      cur = U.chunk;
      bvalid = bidx[g] >= 0;
      v0 = bidx[2 * t] >= 0;
      v1 = bidx[2 * t + 1] >= 0;
    }

    float acc[2][4];
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[m][i] = 0.f;

    if (!mbar_wait_bounded(&sfull[us], uph, abort_flag, A.err)) return;
    const uint8_t* sc = sbuf + us * sslot;
    const uint8_t* brow_s = bbuf + g * bpitch;

    for (int kc = 0; kc < nkc; ++kc) {
      if (!mbar_wait_bounded(&full[s], ph, abort_flag, A.err)) return;
      const int tile = GLU ? kc : 2 * kc + sel;
      if (kb_on && tile < ntiles) {
        const int KB = tile * (IB / 16) + kb;  // global 32-block index along K
        const uint4 b = bvalid ? *reinterpret_cast<const uint4*>(brow_s + KB * 64 + 16 * t)
                               : make_uint4(0, 0, 0, 0);
        const float sc0 = v0 ? exp2i(bexp[(2 * t) * epitch + KB]) : 0.f;
        const float sc1 = v1 ? exp2i(bexp[(2 * t + 1) * epitch + KB]) : 0.f;
        block_mma(acc, stages + s * stage_bytes, q[0], q[1], q[2], q[3],
                  e8m0_to_f32(sc[srows[0] * srow + KB]), e8m0_to_f32(sc[srows[1] * srow + KB]),
                  e8m0_to_f32(sc[srows[2] * srow + KB]), e8m0_to_f32(sc[srows[3] * srow + KB]), b, sc0,
                  sc1);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      if (++s == NS) { s = 0; ph ^= 1; }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sempty[us]);
    if (++us == 2) { us = 0; uph ^= 1; }

    // fixed-order reduction over the warps; red[part][row][col]
    float* r = red + (GLU ? kb : cw) * kRows * kGemvTokens;
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      r[srows[2 * m] * kGemvTokens + 2 * t] = acc[m][0];
      r[srows[2 * m] * kGemvTokens + 2 * t + 1] = acc[m][1];
      r[srows[2 * m + 1] * kGemvTokens + 2 * t] = acc[m][2];
      r[srows[2 * m + 1] * kGemvTokens + 2 * t + 1] = acc[m][3];
    }
    if (!group_barrier(cbar, cph, abort_flag, A.err)) return;
    // epilogue: warp cw < 8 handles chunk column cw, lane = feature f0 + lane
    if (cw < kGemvTokens && bidx[cw] >= 0) {
      const int row = U.r0 + cw;
      if (GLU) {
        float gs = 0.f, us_ = 0.f;
#pragma unroll
        for (int w = 0; w < kParts; ++w) {
          gs += red[(w * kRows + lane) * kGemvTokens + cw];
          us_ += red[(w * kRows + kUnitRows + lane) * kGemvTokens + cw];
        }
        const float av = gs / (1.0f + expf(-gs)) * us_;
        const uint16_t ab = f32_to_bf16(av);
        A.a_out[(size_t)row * A.N + f0 + lane] = ab;
        float qv = bf16_to_f32(ab);
        if (A.actq) qv = mxfp8_roundtrip(qv, mxfp8_block_exp(warp_max(fabsf(qv))));
        const int e = f16_block_exp(warp_max(fabsf(qv)));
        A.ah_out[(size_t)row * A.N + f0 + lane] = __float2half_rn(ldexpf(qv, -e));
        if (lane == 0) A.as_out[(size_t)row * exp_pitch(A.N) + U.fb] = (int8_t)e;
      } else {
        float o = 0.f;
#pragma unroll
        for (int w = 0; w < kParts; ++w) o += red[(w * kRows + lane) * kGemvTokens + cw];
        A.o_out[(size_t)row * A.N + f0 + lane] = o;
      }
    }
    if (!group_barrier(cbar, cph, abort_flag, A.err)) return;
  }
}

struct Geometry {
  int IB, NS;
  size_t smem;
};

template <bool GLU>
Geometry geometry(int K) {
  constexpr int kRows = GLU ? 2 * kUnitRows : kUnitRows;
  constexpr int kParts = GLU ? 8 : 16;
  Geometry g;
  const int rb = K / 2;
  g.IB = (rb % 128 == 0) ? 128 : (rb % 64 == 0) ? 64 : 32;
  const int stage_bytes = (2 * kTileRows * g.IB + 1023) & ~1023;
  g.NS = kStageBudget / stage_bytes;
  if (g.NS > kMaxStages) g.NS = kMaxStages;
  if (g.NS < 2) g.NS = 2;
  const int sbytes = kRows * (K / 32);
  const int sslot = (sbytes + 127) & ~127;
  const int bslot = kGemvTokens * (K * 2 + 64) + kGemvTokens * exp_pitch(K);
  g.smem = (size_t)g.NS * stage_bytes + 2 * (size_t)sslot + ((bslot + 127) & ~127) +
           (size_t)kParts * kRows * kGemvTokens * sizeof(float) + kGemvTokens * sizeof(int) +
           (2 * kMaxStages + 7) * sizeof(uint64_t) + 16 + 1024;  // + alignment slack
  return g;
}

template <bool GLU>
cudaError_t launch_t(ExpertArgs& a, int units_max, cudaStream_t s) {
  const Geometry g = geometry<GLU>(a.K);
  a.IB = g.IB;
  a.NS = g.NS;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(expert_gemv_kernel<GLU>), g.smem);
  if (e != cudaSuccess) return e;
  int grid = num_sms();
  if (units_max < grid) grid = units_max > 0 ? units_max : 1;
  return launch_pdl(expert_gemv_kernel<GLU>, dim3(grid), dim3(kThreads), g.smem, s, a);
}

bool code_map(CUtensorMap* m, const uint8_t* q, int E, int N, int K) {
  const int IB = ((K / 2) % 128 == 0) ? 128 : ((K / 2) % 64 == 0) ? 64 : 32;
  return make_tmap_2d(m, q, 1, (uint64_t)(K / 2), (uint64_t)E * N, (uint64_t)(K / 2), (uint32_t)IB,
                      kTileRows, IB == 128);
}

}  // namespace

cudaError_t launch_expert_glu(const k3moe_dims& d, const k3moe_weights& w, const int32_t* plan,
                              const int32_t* offsets, const int32_t* row_token, const __half* zh,
                              const int8_t* zs, uint16_t* a, __half* ah, int8_t* as, int T,
                              uint32_t* err, cudaStream_t s) {
  (void)offsets;
  ExpertArgs A{};
  if (!code_map(&A.tq0, w.gate_q, d.n_experts, d.inter, d.latent) ||
      !code_map(&A.tq1, w.up_q, d.n_experts, d.inter, d.latent))
    return cudaErrorInvalidValue;
  A.s0 = w.gate_s; A.s1 = w.up_s;
  A.N = d.inter; A.K = d.latent;
  A.plan = plan; A.ctab = plan_ctab(const_cast<int32_t*>(plan), d.n_experts);
  A.row_token = row_token;
  A.brows = T; A.rows_max = T * d.top_k;
  A.bh = zh; A.bs = zs; A.a_out = a; A.ah_out = ah; A.as_out = as;
  A.E = d.n_experts; A.actq = d.actq; A.err = err;
  const int chunks_max = A.rows_max / kGemvTokens + d.n_experts;
  return launch_t<true>(A, chunks_max * (d.inter / kUnitRows), s);
}

cudaError_t launch_expert_down(const k3moe_dims& d, const k3moe_weights& w, const int32_t* plan,
                               const int32_t* offsets, const __half* ah, const int8_t* as,
                               float* o_rows, int T, uint32_t* err, cudaStream_t s) {
  (void)offsets;
  ExpertArgs A{};
  if (!code_map(&A.tq0, w.down_q, d.n_experts, d.latent, d.inter)) return cudaErrorInvalidValue;
  A.s0 = w.down_s;
  A.N = d.latent; A.K = d.inter;
  A.plan = plan; A.ctab = plan_ctab(const_cast<int32_t*>(plan), d.n_experts);
  A.row_token = nullptr;
  A.brows = T * d.top_k; A.rows_max = T * d.top_k;
  A.bh = ah; A.bs = as; A.o_out = o_rows;
  A.E = d.n_experts; A.actq = d.actq; A.err = err;
  const int chunks_max = A.rows_max / kGemvTokens + d.n_experts;
  return launch_t<false>(A, chunks_max * (d.latent / kUnitRows), s);
}

}  // namespace k3moe
