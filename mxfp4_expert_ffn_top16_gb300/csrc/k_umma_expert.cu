// MXFP4 expert FFN for many tokens on block-scaled 5th-generation tensor cores
// (tcgen05.mma kind::mxf8f6f4.block_scale): the weights go into the tensor core as e2m1 codes
// with their e8m0 scales, so no ALU work is spent per weight.
//
// "kimi-k3-in-c", MXFP4 experts: 4-bit codes indexing a 16-entry value table, one 8-bit
// exponent per 32 consecutive weights; "Kimi K3 hardware deep dive", quantisation-aware
// training: MXFP4 weights with MXFP8 activations. For sorted row r of expert e (token t):
//   GLU pass:  a[r] = bf16(silu(G_e z_t) * (U_e z_t))          G_e, U_e [I][L]
//   down pass: o[r] = D_e a[r]                                  D_e [L][I]
//
// Activations enter as e4m3 rows with one e8m0 scale per 32 values (P rows per sorted row):
//   P = 1 (MXFP8 activations): the MXFP8 encoding itself (OCP MX v1.0: shared exponent
//          floor(log2 amax) - 8, E4M3 elements rounded to nearest even, saturating).
//   P = 2 (bf16 activations): hi = E4M3 rounding of v / 2^Xh with Xh = floor(log2 amax) - 7
//          (no saturation: |v| / 2^Xh < 256), lo = v - hi on its own block exponent. bf16 has 8
//          significant bits and each part carries 4, so hi + lo is the bf16 value exactly for
//          every element within 2^-13 of its block maximum; below that the error is under
//          2^-20 of the block maximum. The MMA sees both rows as B columns and the epilogue
//          adds the two results.
//
// Tile: M = 128 weight rows (GLU: 64 gate rows and the 64 up rows of the same features, so
// lane i and lane i + 64 pair up), N = the chunk's activation rows (up to 224: 112 sorted rows
// of bf16 hi + lo pairs, 224 of MXFP8, 192 of MXFP4), K = 128 per pipeline stage (four MMAs of
// K = 32, each with its scale byte; MXFP4: K = 256). Work item = (chunk of one expert's sorted
// rows, feature block), feature block fastest: the CTAs working at one time
// share a chunk's activations and an expert's weights in L2. Each tcgen05 instruction costs
// tens of cycles to issue from the single MMA thread, so N is made as large as tensor memory
// allows (two 224-column accumulators) to keep the tensor pipe, not the issue, the limit.
// Warp 0 (lane 0) loads the packed e2m1 weight tiles (16U4_ALIGN16B tensor map) and the e4m3
// activation tiles, both with the 128-byte swizzle. The stage's scales go into the 32 x 16-byte
// blocks that tcgen05.cp.32x128b.warpx4 copies to tensor memory (lane l, word w = the four
// K-block scales of row 32w + l): the weight rows' block comes with the tiles as one bulk copy
// from a prepared layer's staging image (else warp 10 gathers it with 4-byte cp.async), and warp
// 11 gathers the activation rows' scales the same way; the stage's full barrier counts the bytes
// and one cp.async arrival per gathering lane. Warp 1: tensor-memory owner and MMA issuer, one
// commit per stage. With many tokens the plan lists the experts that received at most 8 rows
// last, and this kernel leaves them to the weights-on-N kernel (big_only).
// Each item accumulates its whole K in one of two tensor-memory slots, so the epilogue of one
// item overlaps the MMAs of the next; eight epilogue warps (two per lane quadrant, one lane = one
// weight row, each half of the sorted rows) drain it and run the epilogue; the GLU epilogue
// transposes through shared memory so each thread quantises one (sorted row, 32-feature block).
#include <cuda_fp16.h>

#include "k3moe_device.cuh"
#include "k3moe_internal.cuh"
#include "k3moe_umma.cuh"

namespace k3moe {
namespace {

constexpr int BM = 128, BKE = 128;        // weight rows, K elements per stage (e4m3 activations)
constexpr int kATile = BM * 128;          // bytes in shared memory: 128-byte rows
// Bytes a stage's weight copy transfers: e4m3 activations (kind::mxf8f6f4) take the weights as
// e2m1 padded to one code per byte in shared memory (K = 128 per stage, 64 packed bytes per row);
// MXFP4 activations (kind::mxf4) take both operands packed, two codes per byte (K = 256 per
// stage in the same 128-byte rows).
template <bool FP4>
constexpr int kAPacked = FP4 ? BM * 128 : BM * 128 / 2;
template <bool FP4>
constexpr int kKStage = FP4 ? 256 : 128;  // K per stage
constexpr int kThreads = 384;             // 0 TMA, 1 MMA, 2-9 epilogue, 10-11 scale gather
constexpr int kEpiWarps = 8;
constexpr int kGather0 = 2 + kEpiWarps;   // first scale-gather warp
constexpr int kAccSlots = 2;
// Tensor-memory scale columns per stage (Cfg::kSfPer). e4m3: A 4, B rows 0..127 4, B rows
// 128..255 4 (one 32-bit word of four K-block scales per row and stage), 16 reserved. MXFP4: two
// words per row and stage (K = 256): A 4 + 4, B 4 + 4 (B rows <= 128); with more than 128 B rows,
// each B word takes 8 columns (rows 0..127, then rows 128..255): 24.
// Scale staging blocks of 32 x 16 bytes per stage (Cfg::kStg): e4m3 A, B rows 0..127, B rows
// 128..255; MXFP4 A word 0, A word 1, B word 0, B word 1 (rows 0..127), then B word 0 and word 1
// of rows 128..255.

// Shapes by chunk size R (sorted rows per item) and activation rows per sorted row P:
// many tokens: R = kUmmaChunkRows with P = 2 (N up to 224), kUmmaChunkRowsWide with MXFP8 (N up
// to 224) or kUmmaChunkRowsFp4 with MXFP4 (N up to 192), four stages each; few tokens:
// R = kGemvTokens (N up to 16, small activation tiles, so eleven stages keep enough weight bytes
// in flight to stream at HBM speed).
template <int R, int P, bool FP4, bool GLU>
struct Cfg {
  static constexpr int kOut = R;                  // sorted rows per item (max)
  static constexpr int kNMax = R == kGemvTokens ? 2 * R : P * R;  // B rows per tile (MMA N <= kNMax)
  static constexpr int kBTile = kNMax * BKE;      // e4m3 (MXFP4: half of it used)
  static constexpr int kStg = FP4 ? (FP4 && P * R > 128 ? 3072 : 2048) : 1536;
  // the down pass has no exchange buffer: a fifth stage fits where its stages are small enough
  static constexpr int kStages =
      R == kGemvTokens ? 11 : (!GLU && 5 * (128 * BKE + kNMax * BKE + kStg) + 1024 + 256 <= 227 * 1024 ? 5 : 4);
  static constexpr bool kWideSf = FP4 && kNMax > 128;  // MXFP4 B scales in two 128-row blocks
  static constexpr int kSfPer = kWideSf ? 24 : 16;
  // the epilogue takes the rows in passes of at most kUmmaChunkRows (its registers and exchange
  // buffer are sized for one pass)
  static constexpr int kPasses = (R + kUmmaChunkRows - 1) / kUmmaChunkRows;
  static constexpr int kRowsPass = R / kPasses;
  static constexpr int kXPitch = kRowsPass + 1;   // GLU exchange row pitch (floats)
  static constexpr uint32_t kSfCol = kAccSlots * kNMax;  // scale columns, kSfPer per stage
  static constexpr uint32_t kTmemCols = R == kGemvTokens ? 256 : 512;
  static_assert(R == kGemvTokens || R == kUmmaChunkRows || R == kUmmaChunkRowsWide || R == kUmmaChunkRowsFp4,
                "chunk size");
  static_assert(R % kPasses == 0 && kRowsPass % 4 == 0, "epilogue passes");
  static_assert(kSfCol + kSfPer * kStages <= kTmemCols, "tensor memory");
  static_assert(kNMax <= 7 * 32, "scale gather groups");
  static_assert(kNMax <= 256 && kNMax % 16 == 0, "MMA N");
};

struct UExpertArgs {
  CUtensorMap ta0;     // GLU: gate codes; down: down codes. {K codes, E*N rows}, box {128, 64|128}
  CUtensorMap ta1;     // GLU: up codes
  CUtensorMap tb;      // activation rows, e4m3 {K, P*rows}, box {128, R*P}
  const uint8_t* s0;   // weight scales [E][N][K/32]
  const uint8_t* s1;   // GLU: up scales
  const uint8_t* sb;   // activation scales [P*rows][exp_pitch(K)]
  int32_t* plan;
  int N, K, E;         // output features per expert, reduction length, experts
  int rows_max;        // sorted rows (T * k)
  uint8_t* aq;         // GLU: quantised output for the down pass [P*rows][N] e4m3
  uint8_t* aqs;        //      its scales [P*rows][exp_pitch(N)]
  float* o_out;        // down: [rows][N] fp32
  int big_only;        // many tokens: only the chunks of the experts with more than kSmallExpertRows rows
  const uint8_t* pw;   // weight scales in the staging image (null: gathered row by row): per tile
                       // row-block (GLU: 64 features, down: 128 rows) and 128-code chunk, 512 bytes
  uint32_t* err;
};

__device__ __forceinline__ void umma_mx(uint32_t d, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t sfa,
                                        uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %6, 0; tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X "
      "[%0], %1, %2, %3, [%4], [%5], p; }" ::"r"(d),
      "l"(ad), "l"(bd), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
      : "memory");
}
// A e2m1, B e4m3, e8m0 scales, fp32 accumulation, both K-major; scale byte kk of each word.
__device__ __forceinline__ uint32_t idesc_mx(int N, int kk) {
  return ((uint32_t)kk << 4) | (5u << 7) | (0u << 10) | ((uint32_t)(N >> 3) << 17) | (1u << 23) |
         ((uint32_t)(BM >> 4) << 24) | ((uint32_t)kk << 29);
}
// kind::mxf4: A and B e2m1 (packed), e8m0 scales, fp32 accumulation, K-major, K = 64 per MMA
// (scale_vec::2X: two scale bytes per row, starting at byte sf of the scale word).
__device__ __forceinline__ uint32_t idesc_mxf4(int N, int sf) {
  return ((uint32_t)sf << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | (1u << 23) |
         ((uint32_t)(BM >> 4) << 24) | ((uint32_t)sf << 29);
}
__device__ __forceinline__ void umma_mxf4(uint32_t d, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t sfa,
                                          uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %6, 0; tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X "
      "[%0], %1, %2, %3, [%4], [%5], p; }" ::"r"(d),
      "l"(ad), "l"(bd), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
      : "memory");
}
// Eight values -> eight e2m1 codes (nearest even, saturating at +-6), packed low nibble first.
__device__ __forceinline__ uint32_t e2m1x8(const float* v) {
  uint32_t r = 0;
#pragma unroll
  for (int i = 0; i < 8; i += 2) {
    uint32_t b;
    asm("{ .reg .b8 t; cvt.rn.satfinite.e2m1x2.f32 t, %1, %2; cvt.u32.u8 %0, t; }" : "=r"(b) : "f"(v[i + 1]), "f"(v[i]));
    r |= b << (4 * i);
  }
  return r;
}
// Shared exponent of an MXFP4 block from its amax (OCP MX v1.0: floor(log2 amax) - 2, clamped to
// the e8m0 range); an all-zero block gets -127.
__device__ __forceinline__ int mxfp4_block_exp(float amax) {
  if (!(amax > 0.0f)) return -127;
  if (!(amax <= 3.4028235e38f)) return 127;
  const int X = ilog2_floor(amax) - 2;
  return X < -127 ? -127 : (X > 127 ? 127 : X);
}

// Descriptor of a 32 x 16-byte scale staging block: no swizzle, 8-row groups 128 bytes apart.
__device__ __forceinline__ uint64_t sdesc_sf(uint32_t addr) {
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)(128 >> 4) << 16) | ((uint64_t)(128 >> 4) << 32) |
         ((uint64_t)1 << 46);
}

// 4-byte asynchronous copy global -> shared (shared-window address).
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
// Arrives on `bar` once every cp.async this thread issued so far has landed (the arrival is
// part of the barrier's expected count: .noinc).
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ float max_in_group4(float v) {
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
  return fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
}

// One 32-value block (v, one thread) -> P rows of 32 E4M3 codes (8 words each) and block
// exponents. P = 2: v is left holding the lo remainders.
template <int P>
__device__ __forceinline__ void quant_block32(float (&v)[32], uint32_t (&codes)[P][8], int (&X)[P]) {
#pragma unroll
  for (int p = 0; p < P; ++p) {
    float am = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) am = fmaxf(am, fabsf(v[i]));
    X[p] = p == 0 ? block_exp<P>(am) : split_block_exp(am);
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
      const uint32_t c01 = e4m3x2(mul_pow2(v[i], -X[p]), mul_pow2(v[i + 1], -X[p]));
      const uint32_t c23 = e4m3x2(mul_pow2(v[i + 2], -X[p]), mul_pow2(v[i + 3], -X[p]));
      codes[p][i / 4] = c01 | (c23 << 16);
      if (P == 2 && p == 0) {  // remainders for the lo row (exact)
        const float2 h01 = e4m3x2_value(c01), h23 = e4m3x2_value(c23);
        v[i] -= mul_pow2(h01.x, X[0]);
        v[i + 1] -= mul_pow2(h01.y, X[0]);
        v[i + 2] -= mul_pow2(h23.x, X[0]);
        v[i + 3] -= mul_pow2(h23.y, X[0]);
      }
    }
  }
}

template <bool GLU, int P, int R, bool FP4>
__global__ void __launch_bounds__(kThreads, 1) umma_expert_kernel(const __grid_constant__ UExpertArgs A) {
  static_assert(!FP4 || P == 1, "MXFP4 activations: one row per sorted row");
  using CF = Cfg<R, P, FP4, GLU>;
  constexpr int kStg = CF::kStg, kSfPerStage = CF::kSfPer;
  constexpr bool kWideSf = CF::kWideSf;
  constexpr int kOut = CF::kOut, kNMax = CF::kNMax, kBTile = CF::kBTile, kStages = CF::kStages;
  constexpr int kXPitch = CF::kXPitch;
  constexpr uint32_t kSfCol = CF::kSfCol, kTmemCols = CF::kTmemCols;
  constexpr int kFB = GLU ? 64 : 128;  // output features per item
  constexpr int kBRows = kOut * P;     // activation rows per tile
  constexpr uint32_t kBTx = kBRows * BKE;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int srow = A.K / 32, spb = exp_pitch(A.K);
  uint8_t* sA = smem;
  uint8_t* sB = sA + kStages * kATile;
  uint8_t* stg = sB + kStages * kBTile;                            // kStages x kStg
  float* xg = reinterpret_cast<float*>(stg + kStages * kStg);  // GLU: [64][kXPitch]
  uint64_t* full = reinterpret_cast<uint64_t*>(xg + (GLU ? 64 * kXPitch : 0));
  uint64_t* empty = full + kStages;
  uint64_t* accf = empty + kStages;
  uint64_t* acce = accf + kAccSlots;
  uint64_t* ebar = acce + kAccSlots;  // epilogue group barrier
  uint64_t* drain = ebar + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      // the expect_tx arrival + one cp.async arrival per gathering lane (weight rows: none when
      // their scales come with the tiles)
      mbar_init(&full[s], 1 + (A.pw ? 32 : 64));
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < kAccSlots; ++b) {
      mbar_init(&accf[b], 1);
      mbar_init(&acce[b], kEpiWarps);
    }
    mbar_init(ebar, kEpiWarps);
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

  // chunk table of the plan for this chunk size (entries {expert, first row, rows, 0})
  const int4* ctab;
  int C;
  if (R != kGemvTokens) {
    ctab = plan_ctab64(A.plan, A.E, A.rows_max) + 1;
    C = A.big_only ? ctab[-1].y : ctab[-1].x;
  } else {
    ctab = plan_ctab(A.plan, A.E);
    C = A.plan[1];
  }
  const int fbs = A.N / kFB;
  const long long cmax = R != kGemvTokens ? plan_ctab64_max(A.E, A.rows_max) : A.rows_max / R + A.E;
  const int items = (C > 0 && C <= cmax) ? C * fbs : 0;
  const int nk = A.K / kKStage<FP4>;

  // item u -> (expert, first sorted row, rows, first feature); false for a corrupt entry
  auto item_of = [&](int u, int& e, int& r0, int& nr, int& f0) -> bool {
    const int c = u / fbs, fb = u - c * fbs;
    const int4 t = ctab[c];
    const bool ok = t.x >= 0 && t.x < A.E && t.y >= 0 && t.z > 0 && t.z <= kOut && t.y + t.z <= A.rows_max;
    e = ok ? t.x : 0;
    r0 = ok ? t.y : 0;
    nr = ok ? t.z : 0;
    f0 = fb * kFB;
    return ok;
  };

  if (warp == 0) {  // ---------------- tile loads
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < items && ok; u += gridDim.x) {
        int e, r0, nr, f0;
        if (!item_of(u, e, r0, nr, f0)) atomicOr(A.err, kErrIndex);
        const int wrow = e * A.N + f0;
        constexpr uint32_t kSfTx = FP4 ? 1024u : 512u;  // the tile's weight-scale blocks per stage
        const size_t pblk = (size_t)(wrow / (GLU ? 64 : 128)) * (A.K / 128);
        for (int kc = 0; kc < nk; ++kc) {
          if (!mbar_wait_bounded(&empty[s], ph ^ 1, abort_flag, A.err)) { ok = false; break; }
          mbar_arrive_expect_tx(&full[s], kAPacked<FP4> + kBTx + (A.pw ? kSfTx : 0u));
          if (A.pw)
            bulk_g2s_stream(stg + s * kStg, A.pw + (pblk + (size_t)kc * (FP4 ? 2 : 1)) * 512, kSfTx, &full[s],
                            l2_evict_first());
          tma_load_2d(sA + s * kATile, &A.ta0, kc * BKE, wrow, &full[s]);
          if (GLU) tma_load_2d(sA + s * kATile + 64 * 128, &A.ta1, kc * BKE, wrow, &full[s]);
          tma_load_2d(sB + s * kBTile, &A.tb, kc * BKE, P * r0, &full[s]);
          if (++s == kStages) { s = 0; ph ^= 1; }
        }
      }
    }
  } else if (warp >= kGather0) {  // ---------------- scale gather: weight rows, then activation rows
    // Activation rows past the chunk are not copied: a B row only affects its own output
    // column, and those columns are never read.
    const bool wa = warp == kGather0;
    int s = 0;
    uint32_t ph = 0;
    bool ok = !(wa && A.pw);  // (the weight scales come with the tiles)
    for (int u = blockIdx.x; u < items && ok; u += gridDim.x) {
      int e, r0, nr, f0;
      item_of(u, e, r0, nr, f0);
      const size_t wrow = (size_t)e * A.N + f0;
      const uint8_t* src[7];
      uint32_t dst[7];
      int n = 0;
      const uint32_t st_lane = smem_u32(stg) + lane * 16;
      if (wa) {
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const int r = 32 * w + lane;
          src[w] = (GLU && r >= 64) ? A.s1 + (wrow + r - 64) * srow : A.s0 + (wrow + r) * srow;
          dst[w] = st_lane + 4 * w;
        }
        n = 4;
      } else if (FP4) {  // word 0 of rows 0..127 in block 2, word 1 in block 3 (rows 128..: 4, 5)
#pragma unroll
        for (int w = 0; w < (kNMax + 31) / 32 && w < 7; ++w) {
          const int rb = 32 * w + lane;
          src[w] = A.sb + ((size_t)r0 + rb) * spb;
          dst[w] = st_lane + (w < 4 ? 1024 + 4 * w : 2048 + 4 * (w - 4));
          if (rb < nr) n = w + 1;
        }
      } else {
#pragma unroll
        for (int w = 0; w < 7; ++w) {
          const int rb = 32 * w + lane;  // B row; block rb / 128 of the stage, word (rb / 32) % 4
          src[w] = A.sb + ((size_t)P * r0 + rb) * spb;
          dst[w] = st_lane + 512 * (1 + (w >> 2)) + 4 * (w & 3);
          if (rb < P * nr) n = w + 1;  // rows of this lane that exist: w < n
        }
      }
      for (int kc = 0; kc < nk; ++kc) {
        if (!mbar_wait_warp(&empty[s], ph ^ 1, abort_flag, A.err)) { ok = false; break; }
        const uint32_t so = (uint32_t)(s * kStg);
        if (FP4) {  // eight K-block scales per row and stage: two words, the second 512 bytes on
#pragma unroll
          for (int w = 0; w < 7; ++w)
            if (w < n) {
              cp_async4(dst[w] + so, src[w] + 8 * kc);
              cp_async4(dst[w] + so + 512, src[w] + 8 * kc + 4);
            }
        } else {
#pragma unroll
          for (int w = 0; w < 7; ++w)
            if (w < n) cp_async4(dst[w] + so, src[w] + 4 * kc);
        }
        cp_async_arrive(&full[s]);
        if (++s == kStages) { s = 0; ph ^= 1; }
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");  // nothing lands after the block has gone
  } else if (warp == 1) {  // ---------------- MMA issue: the whole warp runs the loop, one lane issues
    int s = 0, slot = 0;
    uint32_t ph = 0, aph = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < items && ok; u += gridDim.x) {
      int e, r0, nr, f0;
      item_of(u, e, r0, nr, f0);
      int Nc = P * nr;
      Nc = Nc < 16 ? 16 : ((Nc + 15) & ~15);
      if (!mbar_wait_warp(&acce[slot], aph ^ 1, abort_flag, A.err)) { ok = false; break; }
      const uint32_t d = tmem + (uint32_t)(slot * kNMax);
      for (int kc = 0; kc < nk; ++kc) {
        if (!mbar_wait_warp(&full[s], ph, abort_flag, A.err)) { ok = false; break; }
        // scale columns: A (4), then B rows 0..127 (4) and B rows 128..255 (4)
        const uint32_t tsa = tmem + kSfCol + kSfPerStage * s, tsb = tsa + 4;
        const uint32_t st0 = smem_u32(stg + s * kStg);
        const uint32_t a0 = smem_u32(sA + s * kATile), b0 = smem_u32(sB + s * kBTile);
        if (FP4) {
          // scale columns: A word 0 (4), A word 1 (4), B word 0 (4), B word 1 (4); the MMA of
          // K block pair kk uses word kk / 2, bytes 2 (kk % 2) and 2 (kk % 2) + 1. With more than
          // 128 B rows each B word takes 8 columns, rows 128.. in its upper 4.
          constexpr uint32_t kBw = kWideSf ? 8 : 4;  // columns per B word
          if (elect_one()) {
            fence_async_smem();  // the scales arrived through cp.async; tcgen05.cp reads them
            tc_fence_after();
            asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(tsa), "l"(sdesc_sf(st0)));
            asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(tsa + 4), "l"(sdesc_sf(st0 + 512)));
            asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(tsa + 8),
                         "l"(sdesc_sf(st0 + 1024)));
            asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(tsa + 8 + kBw),
                         "l"(sdesc_sf(st0 + 1536)));
            if (kWideSf && Nc > 128) {
              asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(tsa + 12),
                           "l"(sdesc_sf(st0 + 2048)));
              asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(tsa + 12 + kBw),
                           "l"(sdesc_sf(st0 + 2560)));
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_mxf4(d, sdesc_sw128(a0 + kk * 32), sdesc_sw128(b0 + kk * 32), idesc_mxf4(Nc, 2 * (kk & 1)),
                        tsa + 4 * (kk >> 1), tsa + 8 + kBw * (kk >> 1), (kc | kk) != 0 ? 1u : 0u);
            umma_commit(&empty[s]);
          }
        } else if (elect_one()) {
          fence_async_smem();  // the scales arrived through cp.async; tcgen05.cp reads them
          tc_fence_after();
          asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(tsa), "l"(sdesc_sf(st0)));
          asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(tsb), "l"(sdesc_sf(st0 + 512)));
          if (Nc > 128)
            asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(tsb + 4),
                         "l"(sdesc_sf(st0 + 1024)));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_mx(d, sdesc_sw128(a0 + kk * 32), sdesc_sw128(b0 + kk * 32), idesc_mx(Nc, kk), tsa, tsb,
                    (kc | kk) != 0 ? 1u : 0u);
          umma_commit(&empty[s]);  // tiles and scale block of this stage free again
        }
        __syncwarp();
        if (++s == kStages) { s = 0; ph ^= 1; }
      }
      if (!ok) break;
      if (elect_one()) umma_commit(&accf[slot]);
      __syncwarp();
      if (++slot == kAccSlots) { slot = 0; aph ^= 1; }
    }
    // every issued MMA has completed before the tensor memory is released
    if (elect_one()) {
      umma_commit(drain);
      volatile int no_abort = 0;
      mbar_wait_bounded(drain, 0, &no_abort, A.err);
    }
    __syncwarp();
  } else {  // ---------------- epilogue warps 2..9: lane quadrant q = warp % 4, row half h
    constexpr int kRowsPass = CF::kRowsPass, kPasses = CF::kPasses;
    constexpr int kHalf = kRowsPass / 2;  // sorted rows per epilogue warp and pass
    constexpr int kQ = kHalf / 2;         // GLU exchange split within a half
    const int eq = warp - 2, q = warp & 3, h = eq >> 2;
    const int lrow = q * 32 + lane;       // tile row = tensor-memory lane
    const int et = eq * 32 + lane;        // 0..255 over the epilogue threads
    int slot = 0;
    uint32_t aph = 0, eph = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < items && ok; u += gridDim.x) {
      int e, r0, nr, f0;
      item_of(u, e, r0, nr, f0);
      if (!mbar_wait_warp(&accf[slot], aph, abort_flag, A.err)) { ok = false; break; }
      tc_fence_after();
      for (int pass = 0; pass < kPasses && ok; ++pass) {
      const int pbase = pass * kRowsPass;  // first sorted row of this pass
      const int j0 = pbase + h * kHalf;    // first sorted row of this warp's half
      const int ncols = P * (nr - j0);    // live accumulator columns of this half (may be <= 0)
      float sum[kHalf];
#pragma unroll
      for (int i = 0; i < kHalf; ++i) sum[i] = 0.f;
      const uint32_t base =
          tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(slot * kNMax + P * j0);
#pragma unroll
      for (int c = 0; c < (P * kHalf + 15) / 16; ++c) {
        if (c * 16 < ncols) {  // warp-uniform
          uint32_t v[16];
          tmem_ld16(base + c * 16, v);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16 / P; ++i) {
            if (c * (16 / P) + i < kHalf) {  // compile-time
              float x = __uint_as_float(v[P * i]);
              if (P == 2) x += __uint_as_float(v[P * i + 1]);
              sum[c * (16 / P) + i] += x;
            }
          }
        }
      }
      if (pass == kPasses - 1) {  // the accumulator is free once its last columns are read
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acce[slot]);
      }
      if (GLU) {
        // 1. within each half of the sorted rows, the gate row (lanes 0..63) of feature f parks
        // its sums for the half's upper kQ rows and the up row (lanes 64..127) its sums for the
        // lower kQ rows; 2. each forms a = bf16(silu(gate) * up) for its other quarter in place;
        // 3. every epilogue thread quantises one (sorted row, 32-feature block) of a into P
        // e4m3 rows for the down pass. All rows are handled without a per-row test so the
        // compiler can interleave them; rows past nr hold unused values and are never stored.
        // (a quarter with no row of the chunk is skipped: its values are never read)
        float* xr = xg + (lrow & 63) * kXPitch + (j0 - pbase);
        const bool lo_live = j0 < nr, hi_live = j0 + kQ < nr;  // warp-uniform
        if (q < 2) {
          if (hi_live) {
#pragma unroll
            for (int i = kQ; i < kHalf; ++i) xr[i] = sum[i];
          }
        } else if (lo_live) {
#pragma unroll
          for (int i = 0; i < kQ; ++i) xr[i] = sum[i];
        }
        if (!group_barrier_warp(ebar, eph, abort_flag, A.err)) { ok = false; break; }
        // silu(g) = g / (1 + e^-g) in the fast forms, ~1e-6 relative, far below bf16 rounding
        if (q < 2) {
          if (lo_live) {
#pragma unroll
            for (int i = 0; i < kQ; ++i) {
              const float g = sum[i];
              xr[i] = bf16_to_f32(f32_to_bf16(__fdividef(g, 1.0f + __expf(-g)) * xr[i]));
            }
          }
        } else if (hi_live) {
#pragma unroll
          for (int i = kQ; i < kHalf; ++i) {
            const float g = xr[i];
            xr[i] = bf16_to_f32(f32_to_bf16(__fdividef(g, 1.0f + __expf(-g)) * sum[i]));
          }
        }
        if (!group_barrier_warp(ebar, eph, abort_flag, A.err)) { ok = false; break; }
        // (sorted row, 32-feature block) units: the pass's rows x 2 blocks over the 256 threads
        for (int unit = et; unit < 2 * kRowsPass; unit += 32 * kEpiWarps) {
          const int jl = unit % kRowsPass, b = unit / kRowsPass, jr = pbase + jl;
          if (jr < nr && FP4) {  // MXFP4: 32 e2m1 codes (16 bytes) and the block exponent
            float v[32], am = 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              v[i] = xg[(32 * b + i) * kXPitch + jl];
              am = fmaxf(am, fabsf(v[i]));
            }
            const int X = mxfp4_block_exp(am);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = mul_pow2(v[i], -X);
            const size_t brow = (size_t)(r0 + jr);
            *reinterpret_cast<uint4*>(A.aq + brow * (A.N / 2) + (f0 + 32 * b) / 2) =
                make_uint4(e2m1x8(v), e2m1x8(v + 8), e2m1x8(v + 16), e2m1x8(v + 24));
            A.aqs[brow * exp_pitch(A.N) + (f0 + 32 * b) / 32] = (uint8_t)(X + 127);
          } else if (jr < nr) {
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = xg[(32 * b + i) * kXPitch + jl];
            uint32_t codes[P][8];
            int X[P];
            quant_block32<P>(v, codes, X);
            const int spo = exp_pitch(A.N);
#pragma unroll
            for (int p = 0; p < P; ++p) {
              const size_t brow = (size_t)P * (r0 + jr) + p;
              uint4* dst = reinterpret_cast<uint4*>(A.aq + brow * A.N + f0 + 32 * b);
              dst[0] = make_uint4(codes[p][0], codes[p][1], codes[p][2], codes[p][3]);
              dst[1] = make_uint4(codes[p][4], codes[p][5], codes[p][6], codes[p][7]);
              A.aqs[brow * spo + (f0 + 32 * b) / 32] = (uint8_t)(X[p] + 127);
            }
          }
        }
        if (!group_barrier_warp(ebar, eph, abort_flag, A.err)) { ok = false; break; }
      } else {
#pragma unroll
        for (int i = 0; i < kHalf; ++i)
          if (j0 + i < nr) A.o_out[(size_t)(r0 + j0 + i) * A.N + f0 + lrow] = sum[i];
      }
      }  // pass
      if (++slot == kAccSlots) { slot = 0; aph ^= 1; }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <bool GLU, int P, int R, bool FP4>
constexpr size_t smem_bytes() {
  using CF = Cfg<R, P, FP4, GLU>;
  return 1024 + (size_t)CF::kStages * (kATile + CF::kBTile) + CF::kStages * CF::kStg +
         (GLU ? 64 * CF::kXPitch * 4 : 0) + (2 * CF::kStages + 2 * kAccSlots + 2) * 8 + 16;
}
static_assert(smem_bytes<true, 2, kGemvTokens, false>() <= 227 * 1024 &&
                  smem_bytes<true, 2, kUmmaChunkRows, false>() <= 227 * 1024 &&
                  smem_bytes<true, 1, kUmmaChunkRowsWide, false>() <= 227 * 1024 &&
                  smem_bytes<true, 1, kUmmaChunkRowsFp4, true>() <= 227 * 1024 &&
                  smem_bytes<true, 1, kGemvTokens, true>() <= 227 * 1024,
              "shared memory");

template <bool GLU, int P, int R, bool FP4>
cudaError_t launch_t(UExpertArgs& a, int items_max, cudaStream_t s) {
  const size_t smem = smem_bytes<GLU, P, R, FP4>();
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(umma_expert_kernel<GLU, P, R, FP4>), smem);
  if (e != cudaSuccess) return e;
  int grid = num_sms();
  if (items_max < grid) grid = items_max > 0 ? items_max : 1;
  return launch_pdl(umma_expert_kernel<GLU, P, R, FP4>, dim3(grid), dim3(kThreads), smem, s, a);
}

// P: activation rows per sorted row for e4m3 activations (1 MXFP8, 2 bf16 as hi + lo); P = 0
// selects MXFP4 activations (kind::mxf4, one packed row per sorted row).
template <bool GLU>
cudaError_t launch_pr(UExpertArgs& a, int P, int R, int items_max, cudaStream_t s) {
  if (R == kGemvTokens) {
    if (P == 0) return launch_t<GLU, 1, kGemvTokens, true>(a, items_max, s);
    return P == 1 ? launch_t<GLU, 1, kGemvTokens, false>(a, items_max, s)
                  : launch_t<GLU, 2, kGemvTokens, false>(a, items_max, s);
  }
  if (P == 0)
    return R == kUmmaChunkRowsFp4 ? launch_t<GLU, 1, kUmmaChunkRowsFp4, true>(a, items_max, s) : cudaErrorInvalidValue;
  if (R == kUmmaChunkRowsWide && P == 1) return launch_t<GLU, 1, kUmmaChunkRowsWide, false>(a, items_max, s);
  if (R != kUmmaChunkRows || P != 2) return cudaErrorInvalidValue;
  return launch_t<GLU, 2, kUmmaChunkRows, false>(a, items_max, s);
}

// z[row_token[r]] (bf16) -> P e4m3 rows with e8m0 block scales per sorted row r (P = 0: one
// MXFP4 row of packed e2m1 codes, OCP MX v1.0 conversion: shared exponent floor(log2 amax) - 2,
// elements rounded to nearest even, saturating at +-6). One warp per (sorted row, 256-value
// segment), so every load of a launch is in flight at once; each lane takes 8 consecutive
// values, four lanes one 32-value block.
// slot_row non-null: one warp per (token, 256-value segment) instead; the token's values are
// converted once and stored to the sorted row of each of its k slots (slot_row[t * k + j]).
template <int P>
__global__ void __launch_bounds__(256) quant_rows_kernel(const uint16_t* __restrict__ z,
                                                         const int32_t* __restrict__ row_token, int rows,
                                                         int T, int L, uint8_t* bq, uint8_t* bs, int* cnt,
                                                         int ncnt, uint32_t* err,
                                                         const int32_t* __restrict__ slot_row, int k) {
  pdl_wait();
  pdl_trigger();
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < ncnt; i += blockDim.x) cnt[i] = 0;
  const int lane = threadIdx.x & 31;
  const int segs = (L + 255) / 256;
  const long long wid = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (wid >= (long long)(slot_row ? T : rows) * segs) return;  // warp-uniform
  const int r = (int)(wid / segs), base = (int)(wid % segs) * 256;
  int t = slot_row ? r : (row_token ? row_token[r] : r);
  if (t < 0 || t >= T) {
    if (lane == 0 && base == 0) atomicOr(err, kErrIndex);
    t = 0;
  }
  // the sorted rows the result goes to: r itself, or each slot's row of token t
  const int nout = slot_row ? k : 1;
  auto out_row = [&](int j) -> int {
    if (!slot_row) return r;
    const int o = __ldg(slot_row + (size_t)t * k + j);
    if (o < 0 || o >= rows) {
      if (lane == 0 && base == 0) atomicOr(err, kErrIndex);
      return -1;
    }
    return o;
  };
  const int sp = exp_pitch(L);
  const int col = base + 8 * lane;
  const bool act = col < L;  // L is a multiple of 32: a block is all in or all out
  float v[8];
  if (act) {
    const uint4 w = *reinterpret_cast<const uint4*>(z + (size_t)t * L + col);
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(ww[i] << 16);
      v[2 * i + 1] = __uint_as_float(ww[i] & 0xffff0000u);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = 0.f;
  }
  if constexpr (P == 0) {
    float am = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) am = fmaxf(am, fabsf(v[i]));
    const int X = mxfp4_block_exp(max_in_group4(am));
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = mul_pow2(v[i], -X);
    const uint32_t packed = e2m1x8(v);
    if (act)
      for (int j = 0; j < nout; ++j) {
        const int o = out_row(j);
        if (o < 0) continue;
        *reinterpret_cast<uint32_t*>(bq + (size_t)o * (L / 2) + col / 2) = packed;
        if ((lane & 3) == 0) bs[(size_t)o * sp + col / 32] = (uint8_t)(X + 127);
      }
  } else {
#pragma unroll
  for (int p = 0; p < P; ++p) {
    float am = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) am = fmaxf(am, fabsf(v[i]));
    const int X = p == 0 ? block_exp<P>(max_in_group4(am)) : split_block_exp(max_in_group4(am));
    uint32_t codes[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      codes[i] = e4m3x2(mul_pow2(v[2 * i], -X), mul_pow2(v[2 * i + 1], -X));
      if (P == 2 && p == 0) {  // keep the remainder for the lo row (exact)
        const float2 h = e4m3x2_value(codes[i]);
        v[2 * i] -= mul_pow2(h.x, X);
        v[2 * i + 1] -= mul_pow2(h.y, X);
      }
    }
    if (act)
      for (int j = 0; j < nout; ++j) {
        const int o = out_row(j);
        if (o < 0) continue;
        const size_t row = (size_t)P * o + p;
        *reinterpret_cast<uint2*>(bq + row * L + col) =
            make_uint2(codes[0] | (codes[1] << 16), codes[2] | (codes[3] << 16));
        if ((lane & 3) == 0) bs[row * sp + col / 32] = (uint8_t)(X + 127);
      }
  }
  }
}

}  // namespace

cudaError_t launch_quant_rows(const uint16_t* z, const int32_t* row_token, int rows, int T, int L, int P,
                              uint8_t* bq, uint8_t* bs, int* cnt, int ncnt, uint32_t* err, cudaStream_t s,
                              const int32_t* slot_row, int k) {
  if (rows <= 0) return cudaSuccess;
  const int warps = 8;
  const long long units = (long long)(slot_row ? T : rows) * ((L + 255) / 256);
  const dim3 grid((unsigned)((units + warps - 1) / warps)), block(32 * warps);
  if (P == 0)
    return launch_pdl(quant_rows_kernel<0>, grid, block, 0, s, z, row_token, rows, T, L, bq, bs, cnt, ncnt, err,
                      slot_row, k);
  if (P == 1)
    return launch_pdl(quant_rows_kernel<1>, grid, block, 0, s, z, row_token, rows, T, L, bq, bs, cnt, ncnt, err,
                      slot_row, k);
  return launch_pdl(quant_rows_kernel<2>, grid, block, 0, s, z, row_token, rows, T, L, bq, bs, cnt, ncnt, err,
                    slot_row, k);
}

cudaError_t launch_umma_glu(const k3moe_dims& d, const k3moe_weights& w, int32_t* plan, const uint8_t* bq,
                            const uint8_t* bs, int P, int T, uint8_t* aq, uint8_t* aqs, uint32_t* err,
                            cudaStream_t s, bool big_only, const PackedScales* ps) {
  const int R = umma_chunk_rows(T, P);
  UExpertArgs A{};
  const uint64_t pitch = (uint64_t)d.latent / 2, wrows = (uint64_t)d.n_experts * d.inter;
  const int rows = T * d.top_k;
  if (P == 0) {  // MXFP4 activations: both operands packed, 128-byte boxes of 256 codes per row
    if (!make_tmap_2d(&A.ta0, w.gate_q, 1, pitch, wrows, pitch, 128, 64, true) ||
        !make_tmap_2d(&A.ta1, w.up_q, 1, pitch, wrows, pitch, 128, 64, true) ||
        !make_tmap_2d(&A.tb, bq, 1, (uint64_t)d.latent / 2, (uint64_t)rows, (uint64_t)d.latent / 2, 128, R, true))
      return cudaErrorInvalidValue;
  } else if (!make_tmap_fp4(&A.ta0, w.gate_q, d.latent, wrows, pitch, 64) ||
             !make_tmap_fp4(&A.ta1, w.up_q, d.latent, wrows, pitch, 64) ||
             !make_tmap_2d(&A.tb, bq, 1, (uint64_t)d.latent, (uint64_t)P * rows, (uint64_t)d.latent, BKE, R * P,
                           true)) {
    return cudaErrorInvalidValue;
  }
  A.s0 = w.gate_s; A.s1 = w.up_s; A.sb = bs; A.plan = plan;
  A.N = d.inter; A.K = d.latent; A.E = d.n_experts; A.rows_max = rows;
  A.aq = aq; A.aqs = aqs; A.err = err;
  A.big_only = big_only && R != kGemvTokens;
  A.pw = ps && d.latent % 128 == 0 ? ps->glu : nullptr;
  const int items_max = (rows / R + d.n_experts) * (d.inter / 64);
  return launch_pr<true>(A, P, R, items_max, s);
}

cudaError_t launch_umma_down(const k3moe_dims& d, const k3moe_weights& w, int32_t* plan, const uint8_t* aq,
                             const uint8_t* aqs, int P, int T, float* o_rows, uint32_t* err, cudaStream_t s,
                             bool big_only, const PackedScales* ps) {
  const int R = umma_chunk_rows(T, P);
  UExpertArgs A{};
  const int rows = T * d.top_k;
  const uint64_t pitch = (uint64_t)d.inter / 2, wrows = (uint64_t)d.n_experts * d.latent;
  if (P == 0) {  // MXFP4 activations (see launch_umma_glu)
    if (!make_tmap_2d(&A.ta0, w.down_q, 1, pitch, wrows, pitch, 128, 128, true) ||
        !make_tmap_2d(&A.tb, aq, 1, pitch, (uint64_t)rows, pitch, 128, R, true))
      return cudaErrorInvalidValue;
  } else if (!make_tmap_fp4(&A.ta0, w.down_q, d.inter, wrows, pitch, 128) ||
             !make_tmap_2d(&A.tb, aq, 1, (uint64_t)d.inter, (uint64_t)P * rows, (uint64_t)d.inter, BKE, R * P,
                           true)) {
    return cudaErrorInvalidValue;
  }
  A.s0 = w.down_s; A.sb = aqs; A.plan = plan;
  A.N = d.latent; A.K = d.inter; A.E = d.n_experts; A.rows_max = rows;
  A.o_out = o_rows; A.err = err;
  A.big_only = big_only && R != kGemvTokens;
  A.pw = ps && d.inter % 128 == 0 ? ps->down : nullptr;
  const int items_max = (rows / R + d.n_experts) * (d.latent / 128);
  return launch_pr<false>(A, P, R, items_max, s);
}

}  // namespace k3moe
