// MXFP4 expert FFN for chunks of up to 8 sorted rows on block-scaled tensor cores, with the
// operands placed so that each MMA carries as many weight bytes as possible: the decode kernel
// for chunks of more than 8 activation rows (P = 2 from 5 tokens on), where a 256-wide weight
// side needs half the MMA instructions per weight byte of the 128-wide one. With many tokens it
// also takes the experts that received at most 8 rows (the tail of the many-token chunk table):
// for them it streams the weights far faster than the many-token kernel's wide tiles.
//
// "kimi-k3-in-c", MXFP4 experts: 4-bit codes into a 16-entry table, one 8-bit exponent per 32
// consecutive weights. For sorted row r of expert e (token t):
//   GLU pass:  a[r] = bf16(silu(G_e z_t) * (U_e z_t))          G_e, U_e [I][L]
//   down pass: o[r] = D_e a[r]                                  D_e [L][I]
//
// At decode sizes the layer streams the selected experts' weights once; every tcgen05 or TMA
// instruction costs tens of cycles to issue from one thread, so the weights sit on the N side
// of tcgen05.mma.kind::mxf8f6f4.block_scale (N = 256 weight rows per MMA, e2m1 through a
// 16U4_ALIGN16B tensor map) and the activation rows on the M side (M = 128, e4m3 with e8m0
// scales, P rows per sorted row as in the many-token kernel: P = 2 splits a bf16 value exactly
// into e4m3 hi + lo, P = 1 is MXFP8). Only the first 8 * P of the 128 M rows carry data: each
// stage loads just those rows (2 KB), the stages' activation tiles sit 2 KB apart, and an
// MMA's remaining rows read whatever follows in shared memory (the later tiles, then the weight
// tiles). Row m of the result depends only on row m of A, so those accumulator rows are never read.
//
// Work item = (chunk of up to 8 sorted rows of one expert, feature block): GLU items take 128
// features (B rows 0..127 gate, 128..255 up), down items 256 features. K = 128 per stage.
// Warp 0 (lane 0) loads the weight and activation tiles; warps 2 and 3 gather the stage's
// scales with cp.async into the 32 x 16-byte blocks tcgen05.cp.32x128b.warpx4 copies to tensor
// memory (lane l, word w = the four K-block scales of row 32w + l); warp 1 issues (one elected
// lane of the converged warp). One 256-column accumulator per item; warps 4 and 8 (tensor-memory
// lanes 0..31) each drain half its columns, add the hi and lo rows, and run the epilogue.
//
// One launch can run both passes: the GLU items, then the down items. Persistent CTAs claim
// items from a global counter in that order (the loading thread claims, and passes each claimed
// item to the CTA's other roles through a small shared-memory queue), so an SM that has no third
// GLU item starts on down items while the others finish theirs. A down item needs the GLU output
// of its whole chunk: each epilogue warp counts its finished GLU items per chunk in global memory
// (release), and the down item's loaders wait (acquire, bounded) until the chunk is complete
// before reading its activations. A down item is claimed only after every GLU item has been
// claimed, and only running CTAs claim, each running its items in claim order (holding at most
// one claimed item ahead): every awaited GLU item is therefore running, done or held behind a GLU
// item, and the waits end, however many of the grid's CTAs the GPU can hold at once (other work
// on the GPU may keep some of them from starting at all).
#include <cuda_fp16.h>

#include "k3moe_device.cuh"
#include "k3moe_internal.cuh"
#include "k3moe_umma.cuh"

namespace k3moe {
namespace {

constexpr int BKE = 128;                  // K per stage
constexpr int kNW = 256;                  // weight rows per item (MMA N)
constexpr int kMA = 128;                  // MMA M
constexpr int kRows = kGemvTokens;        // sorted rows per chunk (8)
constexpr int kStages = 5;
constexpr int kBTile = kNW * BKE;         // weight tile in shared memory (e2m1 padded to bytes)
constexpr int kBPacked = kNW * BKE / 2;   // bytes the weight copies transfer
constexpr int kATile = 2 * kRows * BKE;   // activation rows a stage loads (at most 16 x 128 B)
constexpr int kStgBytes = 1536;           // per stage: A scale block, B rows 0..127, B rows 128..255
constexpr int kThreads = 288;             // warps 0 TMA, 1 MMA, 2-3 gather, 4 and 8 epilogue
constexpr int kEpiWarp0 = 4, kEpiWarp1 = 8;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfCol = kNW;          // 12 columns per stage: A 4, B 8
static_assert(kSfCol + 12 * kStages <= kTmemCols, "tensor memory");

struct WnPass {
  CUtensorMap tw0;     // GLU: gate codes, box {128, 128}; down: down codes, box {128, 256}
  CUtensorMap tw1;     // GLU: up codes, box {128, 128}
  CUtensorMap ta;      // down: activation rows e4m3 {K, P*rows}, box {128, 8*P}
  const uint8_t* s0;   // weight scales [E][N][K/32]
  const uint8_t* s1;   // GLU: up scales
  const uint8_t* p0;   // the same scales in the tcgen05.cp staging image (null: gathered row by row):
  const uint8_t* p1;   //   per 128 rows and 128-code chunk, one 512-byte block
  const uint8_t* sa;   // GLU: activation rows per token [T][P][K] e4m3 (gathered by row_token)
  const uint8_t* sb;   // activation scales: GLU [T][P][exp_pitch(K)] per token; down [P*rows][...]
  int N, K;            // output features per expert, reduction length
};

struct UWnArgs {
  WnPass pass[2];      // [0] GLU, [1] down
  int npass;           // 1: the GLU pass only; 2: GLU then down
  int32_t* plan;
  int small_experts;   // chunks: the many-token table's tail (experts with <= kSmallExpertRows rows)
  const int32_t* row_token;  // sorted row -> token (null: activation row r is sorted row r)
  int ntok;            // tokens (T)
  int E;               // experts
  int rows_max;        // T * k
  uint8_t* aq;         // GLU output [P*rows][inter] e4m3 (the down pass's activations)
  uint8_t* aqs;        //   its scales [P*rows][exp_pitch(inter)]
  float* o_out;        // down output [rows][latent] fp32
  int* chunk_done;     // GLU items finished per chunk, times 2 (one count per epilogue warp); zeroed
  int* item_counter;   // items claimed so far; zeroed
  uint32_t* err;
};

constexpr int kQ = 4;  // claimed items in flight from the loading thread to the other roles
// Roles that take each claimed item from the queue: gather warps 2 and 3, the MMA warp and the
// two epilogue warps.
constexpr int kQConsumers = 5;

// Takes the next claimed item from the queue (whole warp): the item, -1 once the items are
// exhausted, -2 if a wait gave up.
__device__ __forceinline__ int queue_pop(uint64_t* qfull, uint64_t* qempty, const int* qitem, int& qs,
                                         uint32_t& qph, volatile int* abort, uint32_t* err) {
  if (!mbar_wait_warp(&qfull[qs], qph, abort, err)) return -2;
  int u = 0;
  if ((threadIdx.x & 31) == 0) {
    u = qitem[qs];
    mbar_arrive(&qempty[qs]);
  }
  u = __shfl_sync(0xffffffffu, u, 0);
  if (++qs == kQ) { qs = 0; qph ^= 1; }
  return u;
}

// Waits (bounded) until the chunk's GLU output is complete; acquire, then the async proxy may
// read it.
__device__ __forceinline__ bool wait_chunk(const int* cnt, int target, volatile int* abort, uint32_t* err) {
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t i = 0;; ++i) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(cnt) : "memory");
    if (v >= target) break;
    if ((i & 15u) == 15u) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        *abort = 1;
        atomicOr(err, kErrTimeout);
        return false;
      }
    }
    __nanosleep(64);
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");
  return true;
}

__device__ __forceinline__ void umma_mx(uint32_t d, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t sfa,
                                        uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %6, 0; tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X "
      "[%0], %1, %2, %3, [%4], [%5], p; }" ::"r"(d),
      "l"(ad), "l"(bd), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
      : "memory");
}
// A e4m3, B e2m1, e8m0 scales, fp32 accumulation, both K-major, M = 128, N = 256; scale byte kk.
__device__ __forceinline__ uint32_t idesc_dec(int kk) {
  return ((uint32_t)kk << 4) | (0u << 7) | (5u << 10) | ((uint32_t)(kNW >> 3) << 17) | (1u << 23) |
         ((uint32_t)(kMA >> 4) << 24) | ((uint32_t)kk << 29);
}
__device__ __forceinline__ uint64_t sdesc_sf(uint32_t addr) {
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)(128 >> 4) << 16) | ((uint64_t)(128 >> 4) << 32) |
         ((uint64_t)1 << 46);
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// 32 values of one thread -> P rows of 32 E4M3 codes with their block exponents (P = 1: MXFP8;
// P = 2: hi and lo, v left holding the lo remainders).
template <int P>
__device__ __forceinline__ void quant32(float* v, uint32_t (&codes)[P][8], int (&X)[P]) {
#pragma unroll
  for (int p = 0; p < P; ++p) {
    float am = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) am = fmaxf(am, fabsf(v[i]));
    X[p] = (P == 1) ? mxfp8_block_exp(am) : split_block_exp(am);
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
      const uint32_t c01 = e4m3x2(mul_pow2(v[i], -X[p]), mul_pow2(v[i + 1], -X[p]));
      const uint32_t c23 = e4m3x2(mul_pow2(v[i + 2], -X[p]), mul_pow2(v[i + 3], -X[p]));
      codes[p][i / 4] = c01 | (c23 << 16);
      if (P == 2 && p == 0) {
        const float2 h01 = e4m3x2_value(c01), h23 = e4m3x2_value(c23);
        v[i] -= mul_pow2(h01.x, X[0]);
        v[i + 1] -= mul_pow2(h01.y, X[0]);
        v[i + 2] -= mul_pow2(h23.x, X[0]);
        v[i + 3] -= mul_pow2(h23.y, X[0]);
      }
    }
  }
}

template <int P>
__global__ void __launch_bounds__(kThreads, 1) umma_wn_kernel(const __grid_constant__ UWnArgs A) {
  constexpr int kARows = kRows * P;           // activation rows a stage loads
  constexpr uint32_t kATx = kARows * BKE;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  // The activation tiles come first: an MMA reads 128 rows (16 KB) from a tile's start, and what
  // follows the last tile is the weight tiles, still inside this block's shared memory.
  uint8_t* sA = smem;                                  // kStages x kATile
  uint8_t* sB = sA + kStages * kATile;                 // kStages x kBTile
  uint8_t* stg = sB + kStages * kBTile;                // kStages x kStgBytes
  uint64_t* full = reinterpret_cast<uint64_t*>(stg + kStages * kStgBytes);
  uint64_t* empty = full + kStages;
  uint64_t* accf = empty + kStages;
  uint64_t* acce = accf + 1;
  uint64_t* drain = acce + 1;
  uint64_t* qfull = drain + 1;
  uint64_t* qempty = qfull + kQ;
  int* qitem = reinterpret_cast<int*>(qempty + kQ);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(qitem + kQ);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1 + 64);  // the expect_tx arrival + one cp.async arrival per gathering lane
      mbar_init(&empty[s], 1);
    }
    mbar_init(accf, 1);
    mbar_init(acce, 2);
    mbar_init(drain, 1);
    for (int q = 0; q < kQ; ++q) {
      mbar_init(&qfull[q], 1);
      mbar_init(&qempty[q], kQConsumers);
    }
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

  const int4* ctab = plan_ctab(A.plan, A.E);
  int C0 = A.plan[1];
  if (A.small_experts) {
    const int4* t64 = plan_ctab64(A.plan, A.E, A.rows_max);
    const int4 h = t64[0];  // {chunks, chunks of the experts with more rows (listed first), ...}
    const bool hok = h.y >= 0 && h.x >= h.y && h.x <= plan_ctab64_max(A.E, A.rows_max);
    ctab = t64 + 1 + (hok ? h.y : 0);
    C0 = hok ? h.x - h.y : 0;
  }
  const int C = (C0 > 0 && C0 <= A.rows_max / kRows + A.E) ? C0 : 0;
  const int fbs_g = A.pass[0].N / (kNW / 2), fbs_d = A.pass[1].N / kNW;
  const int items_g = C * fbs_g;
  const int items = items_g + (A.npass == 2 ? C * fbs_d : 0);
  const int glu_target = 2 * fbs_g;  // epilogue-warp arrivals that complete a chunk

  // item u: GLU items first (chunk-major), then down items
  struct Item {
    bool glu;
    int c, e, r0, nr, f0;
  };
  auto item_of = [&](int u, Item& it) -> bool {
    it.glu = u < items_g;
    const int fbs = it.glu ? fbs_g : fbs_d;
    const int v = it.glu ? u : u - items_g;
    it.c = v / fbs;
    const int fb = v - it.c * fbs;
    const int4 t = ctab[it.c];
    const bool ok = t.x >= 0 && t.x < A.E && t.y >= 0 && t.z > 0 && t.z <= kRows && t.y + t.z <= A.rows_max;
    it.e = ok ? t.x : 0;
    it.r0 = ok ? t.y : 0;
    it.nr = ok ? t.z : 0;
    it.f0 = fb * (it.glu ? kNW / 2 : kNW);
    return ok;
  };

  if (warp == 0) {  // ---------------- item claims and tile loads
    if (lane == 0) {
      int s = 0, qs = 0;
      uint32_t ph = 0, qph = 0;
      bool ok = true;
      // One claim ahead: the next item is claimed before this one's loads are issued, so the
      // claim's round trip overlaps them. A CTA holds at most one unstarted item, claimed after
      // its current one: a held GLU item sits behind a GLU item, which never waits, so every
      // claimed GLU item still gets run.
      int next = atomicAdd(A.item_counter, 1);
      const uint64_t pol = l2_evict_first();
      while (ok) {
        const int u = next < items ? next : -1;
        if (!mbar_wait_bounded(&qempty[qs], qph ^ 1, abort_flag, A.err)) break;
        qitem[qs] = u;
        mbar_arrive(&qfull[qs]);
        if (++qs == kQ) { qs = 0; qph ^= 1; }
        if (u < 0) break;
        next = atomicAdd(A.item_counter, 1);
        Item it;
        if (!item_of(u, it)) atomicOr(A.err, kErrIndex);
        const WnPass& W = A.pass[it.glu ? 0 : 1];
        const int wrow = it.e * W.N + it.f0;
        const int nk = W.K / BKE;
        // staging blocks of the item's rows 0..127 and 128..255 (GLU: the gate and the up rows)
        const size_t pb0 = (size_t)(wrow / 128) * (W.K / 128), pb1 = it.glu ? pb0 : pb0 + W.K / 128;
        const uint32_t sbytes = W.p0 ? 1024u : 0u;
        // a down item's activations are the GLU output of its chunk
        if (!it.glu && !wait_chunk(A.chunk_done + it.c, glu_target, abort_flag, A.err)) break;
        for (int kc = 0; kc < nk; ++kc) {
          if (!mbar_wait_bounded(&empty[s], ph ^ 1, abort_flag, A.err)) { ok = false; break; }
          if (it.glu) {  // the gather warps copy the GLU activation rows
            mbar_arrive_expect_tx(&full[s], kBPacked + sbytes);
            tma_load_2d_stream(sB + s * kBTile, &W.tw0, kc * BKE, wrow, &full[s], pol);
            tma_load_2d_stream(sB + s * kBTile + (kNW / 2) * 128, &W.tw1, kc * BKE, wrow, &full[s], pol);
          } else {
            mbar_arrive_expect_tx(&full[s], kBPacked + kATx + sbytes);
            tma_load_2d_stream(sB + s * kBTile, &W.tw0, kc * BKE, wrow, &full[s], pol);
            tma_load_2d(sA + s * kATile, &W.ta, kc * BKE, P * it.r0, &full[s]);
          }
          if (W.p0) {  // the weights' scale blocks, next to the activation scales' block
            bulk_g2s_stream(stg + s * kStgBytes + 512, W.p0 + (pb0 + kc) * 512, 512u, &full[s], pol);
            bulk_g2s_stream(stg + s * kStgBytes + 1024, (it.glu ? W.p1 : W.p0) + (pb1 + kc) * 512, 512u, &full[s],
                            pol);
          }
          if (++s == kStages) { s = 0; ph ^= 1; }
        }
      }
    }
  } else if (warp == 2 || warp == 3) {  // ---------------- scale gather
    // warp 2: activation rows (lanes < 8P, word 0) and weight rows 0..127; warp 3: weight rows
    // 128..255 (GLU: the up rows). For GLU items the two warps also copy the activation tile:
    // 8P rows x 128 bytes per stage, 16 bytes per copy, into the 128-byte swizzled layout the
    // MMA reads (16-byte unit j of row m at unit j ^ (m & 7)); rows past the chunk are left out.
    const bool w2 = warp == 2;
    const int gl = lane + (w2 ? 0 : 32);  // 0..63 over the two warps
    int s = 0, qs = 0;
    uint32_t ph = 0, qph = 0;
    bool ok = true;
    while (ok) {
      const int u = queue_pop(qfull, qempty, qitem, qs, qph, abort_flag, A.err);
      if (u < 0) break;
      Item it;
      item_of(u, it);
      const WnPass& W = A.pass[it.glu ? 0 : 1];
      const int srow = W.K / 32, spb = exp_pitch(W.K), nk = W.K / BKE;
      const size_t wrow = (size_t)it.e * W.N + it.f0;
      const uint8_t* ws[4];
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const int r = 32 * w + lane + (w2 ? 0 : 128);  // weight row of the item
        ws[w] = (it.glu && r >= kNW / 2) ? W.s1 + (wrow + r - kNW / 2) * srow : W.s0 + (wrow + r) * srow;
      }
      const bool act = w2 && lane < P * it.nr;
      // token of a sorted row (checked: a bad one reads token 0 and sets the error word)
      auto token = [&](int r) -> size_t {
        const int t = A.row_token ? __ldg(A.row_token + r) : r;
        if (t >= 0 && t < A.ntok) return (size_t)t;
        atomicOr(A.err, kErrIndex);
        return 0;
      };
      // activation row m = lane (scales): a sorted row of the down pass, a token's row of the GLU
      const size_t arow = !act ? 0 : it.glu ? token(it.r0 + lane / P) * P + lane % P : (size_t)P * it.r0 + lane;
      const uint8_t* as = W.sb + arow * spb;
      const uint32_t st_lane = smem_u32(stg) + lane * 16;
      // GLU activation tile: units gl and gl + 64 (row m = unit / 8, 16-byte column j = unit % 8)
      const uint8_t* asrc[2];
      uint32_t adst[2];
      bool aon[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int unit = gl + 64 * h, m = unit >> 3, j = unit & 7;
        aon[h] = it.glu && m < P * it.nr;
        const size_t tr = aon[h] ? token(it.r0 + m / P) * P + m % P : 0;
        asrc[h] = W.sa + tr * W.K + 16 * j;
        adst[h] = smem_u32(sA) + (uint32_t)(m * 128 + ((j ^ (m & 7)) << 4));
      }
      if (!it.glu && w2) {  // the activation scales come from this chunk's GLU items
        int good = 1;
        if (lane == 0) good = wait_chunk(A.chunk_done + it.c, glu_target, abort_flag, A.err) ? 1 : 0;
        good = __shfl_sync(0xffffffffu, good, 0);
        __syncwarp();
        if (!good) { ok = false; break; }
      }
      for (int kc = 0; kc < nk; ++kc) {
        if (!mbar_wait_warp(&empty[s], ph ^ 1, abort_flag, A.err)) { ok = false; break; }
        const uint32_t so = st_lane + (uint32_t)(s * kStgBytes);
#pragma unroll
        for (int h = 0; h < 2; ++h)
          if (aon[h]) cp_async16(adst[h] + (uint32_t)(s * kATile), asrc[h] + (size_t)kc * BKE);
        if (act) cp_async4(so, as + 4 * kc);
        if (!W.p0)  // (else the loading thread copies the weights' scale blocks)
#pragma unroll
          for (int w = 0; w < 4; ++w) cp_async4(so + 512 * (w2 ? 1 : 2) + 4 * w, ws[w] + 4 * kc);
        cp_async_arrive(&full[s]);
        if (++s == kStages) { s = 0; ph ^= 1; }
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");  // nothing lands after the block has gone
  } else if (warp == 1) {  // ---------------- MMA issue (converged warp, one elected lane)
    int s = 0, qs = 0;
    uint32_t ph = 0, aph = 0, qph = 0;
    bool ok = true;
    while (ok) {
      const int u = queue_pop(qfull, qempty, qitem, qs, qph, abort_flag, A.err);
      if (u < 0) break;
      const int nk = A.pass[u < items_g ? 0 : 1].K / BKE;
      if (!mbar_wait_warp(acce, aph ^ 1, abort_flag, A.err)) { ok = false; break; }
      for (int kc = 0; kc < nk; ++kc) {
        if (!mbar_wait_warp(&full[s], ph, abort_flag, A.err)) { ok = false; break; }
        const uint32_t tsa = tmem + kSfCol + 12 * s, tsb = tsa + 4;
        const uint32_t st0 = smem_u32(stg + s * kStgBytes);
        const uint32_t a0 = smem_u32(sA + s * kATile), b0 = smem_u32(sB + s * kBTile);
        if (elect_one()) {
          fence_async_smem();  // the scales arrived through cp.async; tcgen05.cp reads them
          tc_fence_after();
          asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(tsa), "l"(sdesc_sf(st0)));
          asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(tsb), "l"(sdesc_sf(st0 + 512)));
          asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(tsb + 4), "l"(sdesc_sf(st0 + 1024)));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_mx(tmem, sdesc_sw128(a0 + kk * 32), sdesc_sw128(b0 + kk * 32), idesc_dec(kk), tsa, tsb,
                    (kc | kk) != 0 ? 1u : 0u);
          umma_commit(&empty[s]);
        }
        __syncwarp();
        if (++s == kStages) { s = 0; ph ^= 1; }
      }
      if (!ok) break;
      if (elect_one()) umma_commit(accf);
      __syncwarp();
      aph ^= 1;
    }
    if (elect_one()) {  // every issued MMA has completed before the tensor memory is released
      umma_commit(drain);
      volatile int no_abort = 0;
      mbar_wait_bounded(drain, 0, &no_abort, A.err);
    }
    __syncwarp();
  } else if (warp == kEpiWarp0 || warp == kEpiWarp1) {  // ---------------- epilogue (lanes 0..31)
    // Accumulator lane m = activation row m (sorted row m / P, part m % P); column n = weight
    // row n of the item. This warp takes columns [h * 128, h * 128 + 128): for the GLU the gate
    // columns of its 64 features and the matching up columns.
    const int h = warp == kEpiWarp1 ? 1 : 0;
    int qs = 0;
    uint32_t aph = 0, qph = 0;
    for (;;) {
      const int u = queue_pop(qfull, qempty, qitem, qs, qph, abort_flag, A.err);
      if (u < 0) break;
      Item it;
      item_of(u, it);
      if (!mbar_wait_warp(accf, aph, abort_flag, A.err)) break;
      aph ^= 1;
      tc_fence_after();
      float v[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int col =
            it.glu ? (c < 2 ? 64 * h + 32 * c : kNW / 2 + 64 * h + 32 * (c - 2)) : 128 * h + 32 * c;
        uint32_t r[32];
        tmem_ld32(tmem + (uint32_t)col, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) v[32 * c + i] = __uint_as_float(r[i]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acce);  // the accumulator may be overwritten now
      if (P == 2) {  // lane 2j holds the hi part of sorted row j, lane 2j + 1 the lo part
#pragma unroll
        for (int i = 0; i < 128; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i], 1);
      }
      const int jr = lane / P;
      const bool mine = (lane % P) == 0 && jr < it.nr;
      if (it.glu) {
        // v[0..63] gate, v[64..127] up of features f0 + 64h + i; one 32-feature block at a time
        const int N = A.pass[0].N, spo = exp_pitch(N);
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          float a[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float g = v[32 * b + i];  // silu(g) = g / (1 + e^-g), fast forms (~1e-6 relative)
            a[i] = bf16_to_f32(f32_to_bf16(__fdividef(g, 1.0f + __expf(-g)) * v[64 + 32 * b + i]));
          }
          if (mine) {
            uint32_t codes[P][8];
            int X[P];
            quant32<P>(a, codes, X);
            const int f = it.f0 + 64 * h + 32 * b;
#pragma unroll
            for (int p = 0; p < P; ++p) {
              const size_t brow = (size_t)P * (it.r0 + jr) + p;
              uint4* dst = reinterpret_cast<uint4*>(A.aq + brow * N + f);
              dst[0] = make_uint4(codes[p][0], codes[p][1], codes[p][2], codes[p][3]);
              dst[1] = make_uint4(codes[p][4], codes[p][5], codes[p][6], codes[p][7]);
              A.aqs[brow * spo + f / 32] = (uint8_t)(X[p] + 127);
            }
          }
        }
        if (A.npass == 2) {  // publish this warp's part of the chunk's GLU output (release)
          __syncwarp();
          if (lane == 0) {
            asm volatile("fence.proxy.async.global;" ::: "memory");
            __threadfence();
            atomicAdd(A.chunk_done + it.c, 1);
          }
        }
      } else if (mine) {
        float4* dst = reinterpret_cast<float4*>(A.o_out + (size_t)(it.r0 + jr) * A.pass[1].N + it.f0 + 128 * h);
#pragma unroll
        for (int i = 0; i < 32; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
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

constexpr size_t kSmem = 1024 + (size_t)kStages * (kBTile + kATile + kStgBytes) + (2 * kStages + 3 + 2 * kQ) * 8 +
                         kQ * 4 + 16;
static_assert((size_t)kStages * kATile + kBTile >= (size_t)(kStages - 1) * kATile + kMA * BKE,
              "an MMA's 128-row read of the last activation tile stays inside shared memory");
static_assert(kATile % 1024 == 0 && (kStages * kATile) % 1024 == 0, "128-byte swizzle alignment");
static_assert(kSmem <= 227 * 1024, "shared memory");

template <int P>
cudaError_t launch_t(UWnArgs& a, int items_max, cudaStream_t s) {
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(umma_wn_kernel<P>), kSmem);
  if (e != cudaSuccess) return e;
  int grid = num_sms();  // one CTA per SM (the shared memory allows no second)
  if (items_max < grid) grid = items_max > 0 ? items_max : 1;
  return launch_pdl(umma_wn_kernel<P>, dim3(grid), dim3(kThreads), kSmem, s, a);
}

}  // namespace

cudaError_t launch_umma_wn(const k3moe_dims& d, const k3moe_weights& w, const PackedScales* ps, int32_t* plan,
                           const uint8_t* zq, const uint8_t* zqs, const int32_t* row_token, int P, int T,
                           uint8_t* aq, uint8_t* aqs, bool with_down, float* o_rows, int* chunk_done,
                           uint32_t* err, cudaStream_t s, bool small_experts) {
  UWnArgs A{};
  const int rows = T * d.top_k;
  WnPass& G = A.pass[0];
  const uint64_t pitch = (uint64_t)d.latent / 2, wrows = (uint64_t)d.n_experts * d.inter;
  if (!make_tmap_fp4(&G.tw0, w.gate_q, d.latent, wrows, pitch, kNW / 2) ||
      !make_tmap_fp4(&G.tw1, w.up_q, d.latent, wrows, pitch, kNW / 2))
    return cudaErrorInvalidValue;
  G.s0 = w.gate_s; G.s1 = w.up_s; G.sa = zq; G.sb = zqs;
  if (ps) { G.p0 = ps->gate; G.p1 = ps->up; }
  G.N = d.inter; G.K = d.latent;
  int items_max = (rows / kRows + d.n_experts) * (d.inter / (kNW / 2));
  A.npass = 1;
  if (with_down) {
    WnPass& D = A.pass[1];
    if (!make_tmap_fp4(&D.tw0, w.down_q, d.inter, (uint64_t)d.n_experts * d.latent, (uint64_t)d.inter / 2, kNW) ||
        !make_tmap_2d(&D.ta, aq, 1, (uint64_t)d.inter, (uint64_t)P * rows, (uint64_t)d.inter, BKE, kRows * P, true))
      return cudaErrorInvalidValue;
    D.s0 = w.down_s; D.sb = aqs;
    if (ps) D.p0 = ps->down;
    D.N = d.latent; D.K = d.inter;
    items_max += (rows / kRows + d.n_experts) * (d.latent / kNW);
    A.npass = 2;
  } else {
    A.pass[1].N = kNW;  // unused; keeps the item arithmetic defined
    A.pass[1].K = BKE;
  }
  A.plan = plan; A.row_token = row_token; A.ntok = row_token ? T : rows; A.E = d.n_experts; A.rows_max = rows;
  A.small_experts = small_experts ? 1 : 0;
  A.aq = aq; A.aqs = aqs; A.o_out = o_rows; A.chunk_done = chunk_done; A.err = err;
  A.item_counter = chunk_done + plan_chunks_max(d, T);
  return P == 1 ? launch_t<1>(A, items_max, s) : launch_t<2>(A, items_max, s);
}

}  // namespace k3moe
