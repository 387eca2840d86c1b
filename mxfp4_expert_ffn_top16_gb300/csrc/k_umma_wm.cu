// MXFP4 expert FFN for decode (chunks of up to 8 sorted rows) on block-scaled tensor cores, the
// weights on the MMA's M side and the few activation rows on N.
//
// "kimi-k3-in-c", MXFP4 experts: 4-bit codes into a 16-entry table, one 8-bit exponent per 32
// consecutive weights. For sorted row r of expert e (token t):
//   GLU pass:  a[r] = bf16(silu(G_e z_t) * (U_e z_t))          G_e, U_e [I][L]
//   down pass: o[r] = D_e a[r]                                  D_e [L][I]
//
// At decode sizes the layer streams the selected experts' weights once, so the kernel is a
// read stream at the HBM rate with the MMAs riding along. Each tcgen05.mma.kind::mxf8f6f4
// .block_scale takes 128 weight rows on M (e2m1 through a 16U4_ALIGN16B tensor map) and 16
// activation rows on N (e4m3 with e8m0 scales, P rows per sorted row: P = 2 splits a bf16 value
// exactly into e4m3 hi + lo, P = 1 is MXFP8; 8 sorted rows at most, rows past the chunk's are
// never read back). The tensor pipe then does 1/8 of the work a 256-wide weight side would
// (M = 128 is the smallest block-scaled M), and a stage's weight load covers 128 rows x 256
// codes: 128 contiguous bytes per row, the granularity HBM streams well at.
//
// Work item = (chunk of up to 8 sorted rows of one expert, block of 128 weight rows): GLU items
// take 128 features (stages alternate between the gate and the up rows over the same K range,
// into two accumulators), down items 128 output features. K per stage = 128 * cps (cps = 2
// chunks of 128 when the pass's K is a multiple of 256, else 1).
// Warp 0 (lane 0) claims items and loads the weight tiles (and a down item's activation tile);
// the weights' scales go to tensor memory through tcgen05.cp.32x128b.warpx4 from 32 x 16-byte
// blocks (lane l, word w = four K-block scales of row 32w + l): with the scales repacked into
// that image beforehand (k3moe_layer_init), the loading thread bulk-copies a stage's blocks along
// with its weight tile; otherwise warps 2 and 3 gather them with cp.async. Warps 2 and 3 also
// gather the activation rows' scales and, for GLU items, the chunk's activation rows; warp 1 issues (one elected lane of the
// converged warp); warps 4..7 (tensor-memory lanes 32q..32q+31) each drain 32 weight rows of the
// item's accumulator and run the epilogue. Two accumulator buffers: the next item's MMAs start
// while the epilogue still reads the last one.
//
// For one token the kernel can also do the routing: after the grid dependency wait every CTA
// selects the token's experts from the router logits (the same block-wide selection as the
// routing kernel) and keeps the plan in shared memory (chunk c = selected expert c, sorted row
// c); CTA 0 also writes the routing outputs. That saves a launch, its hand-off and the plan's
// round trip through global memory.
//
// One launch runs both passes: the GLU items, then the down items. Persistent CTAs claim items
// from a global counter in that order (the loading thread claims, one item ahead, and passes each
// claimed item to the CTA's other roles through a small shared-memory queue), so an SM that has
// no further GLU item starts on down items while the others finish theirs. A down item needs the
// GLU output of its whole chunk: each epilogue warp counts its finished GLU items per chunk in
// global memory (release); a down item's weight loads for the first stages go out at once, and
// its activation loads wait (acquire, bounded) until the chunk is complete. A down item is
// claimed only after every GLU item has been claimed, and only running CTAs claim, each running
// its items in claim order (holding at most one claimed item ahead): every awaited GLU item is
// therefore running, done or held behind a GLU item, and the waits end, however many of the
// grid's CTAs the GPU can hold at once.
#include <cuda_fp16.h>

#include "k3moe_device.cuh"
#include "k3moe_internal.cuh"
#include "k3moe_select.cuh"
#include "k3moe_umma.cuh"

namespace k3moe {
namespace {

constexpr int kMW = 128;                  // weight rows per MMA and per item (M)
constexpr int kNA = 16;                   // MMA N: the chunk's activation rows (8 x P), padded
constexpr int kRows = kGemvTokens;        // sorted rows per chunk (8)
constexpr int kChunkA = kMW * 128;        // one 128-code chunk of 128 weight rows in shared memory (16 KB)
constexpr int kATile = 2 * kChunkA;       // per stage, room for two chunks
constexpr int kSfBytes = 2048;            // per stage: SFA blocks (K-blocks 0-3, 4-7), then SFB blocks
constexpr int kQ = 4;  // claimed items in flight from the loading thread to the other roles
// Shared-memory shape for RB activation rows held per chunk. The MMA reads N = 16 rows; with
// RB = 8 (a chunk carries at most 8 activation rows: P = 1, or P = 2 with at most 4 tokens) its
// rows 8..15 read whatever follows (the next chunk's tile, or the scale area), and the columns
// they produce are never read back. The 2 KB saved per stage buy a sixth stage: more weight
// bytes in flight to the SM.
template <int RB>
struct WmShape {
  static constexpr int kStages = RB == 8 ? 6 : 5;
  static constexpr int kChunkB = RB * 128;  // one 128-byte chunk of the RB activation rows
  static constexpr int kBTile = 2 * kChunkB;
  static constexpr size_t kSmem =
      1024 + (size_t)kStages * (kATile + kBTile + kSfBytes) + (2 * kStages + 5 + 2 * kQ) * 8 + kQ * 4 + 16;
  static_assert(kBTile % 1024 == 0 && kChunkB % 1024 == 0, "128-byte swizzle alignment");
  static_assert(kSmem <= 227 * 1024, "shared memory");
};
constexpr int kThreads = 256;             // warps 0 TMA, 1 MMA, 2-3 gather, 4-7 epilogue
constexpr int kEpiWarp0 = 4;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kAccCols = 32;         // per buffer: GLU gate at +0, up at +16; down at +0
constexpr uint32_t kSfCol = 2 * kAccCols; // 16 columns per stage: SFA 0..7, SFB 8..15
static_assert(kSfCol + 16 * WmShape<8>::kStages <= kTmemCols, "tensor memory");

struct WmPass {
  CUtensorMap tw0;     // GLU: gate codes; down: down codes. {128 codes, rows, K/128 chunks}, box {128, 128, cps}
  CUtensorMap tw1;     // GLU: up codes
  CUtensorMap ta;      // down: activation rows e4m3 {128, P*rows, K/128}, box {128, 16, cps}
  const uint8_t* s0;   // weight scales [E][N][K/32]
  const uint8_t* s1;   // GLU: up scales
  const uint8_t* p0;   // the same scales in the staging image (null: gathered from s0 / s1 instead):
  const uint8_t* p1;   //   per 128 rows and 128-code chunk, the 512-byte block tcgen05.cp copies
  const uint8_t* sa;   // GLU: activation rows per token [T][P][K] e4m3 (gathered by row_token)
  const uint8_t* sb;   // activation scales: GLU [T][P][exp_pitch(K)] per token; down [P*rows][...]
  int N, K, cps;       // output features per expert, reduction length, 128-chunks per stage
};

struct UWmArgs {
  WmPass pass[2];      // [0] GLU, [1] down
  int32_t* plan;
  const int32_t* row_token;  // sorted row -> token
  int ntok;            // tokens (T)
  int E;               // experts
  int rows_max;        // T * k
  uint8_t* aq;         // GLU output [P*rows][inter] e4m3 (the down pass's activations)
  uint8_t* aqs;        //   its scales [P*rows][exp_pitch(inter)]
  float* o_out;        // down output [rows][latent] fp32
  int* chunk_done;     // GLU items finished per chunk, times 4 (one count per epilogue warp); zeroed
  int* item_counter;   // items claimed so far; zeroed
  DecodeSelect sel;    // logits non-null: one token, the kernel selects its experts (see launch_umma_decode)
  int k;
  uint32_t* err;
};

// This CTA's share of [p, p + bytes) into L2 with bulk prefetches (bytes a multiple of 256, p
// 16-byte aligned); the lines keep the normal eviction priority, above the streamed weights'.
__device__ __forceinline__ void l2_fetch_slice(const void* p, long long bytes) {
  const long long per = (bytes / gridDim.x + 255) / 256 * 256;
  const long long b0 = per * blockIdx.x;
  const long long b1 = b0 + per < bytes ? b0 + per : bytes;
  for (long long b = b0; b < b1; b += 32768) {
    const uint32_t n = (uint32_t)(b1 - b < 32768 ? b1 - b : 32768);
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(static_cast<const uint8_t*>(p) + b), "r"(n)
                 : "memory");
  }
}

// Roles that take each claimed item from the queue: gather warps 2 and 3, the MMA warp and the
// four epilogue warps.
constexpr int kQConsumers = 7;

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
// A e2m1 (weights), B e4m3 (activations), e8m0 scales, fp32 accumulation, both K-major,
// M = 128, N = 16; scale byte q of the A and B scale words.
__device__ __forceinline__ uint32_t idesc_wm(int q) {
  return ((uint32_t)q << 4) | (5u << 7) | (0u << 10) | ((uint32_t)(kNA >> 3) << 17) | (1u << 23) |
         ((uint32_t)(kMW >> 4) << 24) | ((uint32_t)q << 29);
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
// One E4M3 code of v * 2^-X (round to nearest even, saturating).
__device__ __forceinline__ uint32_t e4m3_code(float v, int X) { return e4m3x2(mul_pow2(v, -X), 0.f) & 0xffu; }

template <int P, int RB>
__global__ void __launch_bounds__(kThreads, 1) umma_wm_kernel(const __grid_constant__ UWmArgs A) {
  constexpr int kStages = WmShape<RB>::kStages, kChunkB = WmShape<RB>::kChunkB, kBTile = WmShape<RB>::kBTile;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sA = smem;                                  // kStages x kATile (weights)
  uint8_t* sB = sA + kStages * kATile;                 // kStages x kBTile (activation rows)
  uint8_t* stg = sB + kStages * kBTile;                // kStages x kSfBytes
  uint64_t* full = reinterpret_cast<uint64_t*>(stg + kStages * kSfBytes);
  uint64_t* empty = full + kStages;
  uint64_t* accf = empty + kStages;   // [2]
  uint64_t* acce = accf + 2;          // [2]
  uint64_t* drain = acce + 2;
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
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accf[b], 1);
      mbar_init(&acce[b], 4);
    }
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
  if (A.sel.l2_next_bytes > 0 && threadIdx.x == 64) l2_fetch_slice(A.sel.l2_next, A.sel.l2_next_bytes);

  __shared__ int4 s_ctab[32];
  const int4* ctab;
  int C;
  if (A.sel.logits) {  // one token: select its experts here (all 256 threads)
    const int own_e = block_topk(A.sel.logits, 0, A.E, A.k, A.sel.idx, A.sel.wts, blockIdx.x == 0);
    if (threadIdx.x < A.k) s_ctab[threadIdx.x] = make_int4(own_e, threadIdx.x, 1, 0);
    if (blockIdx.x == 0)  // (CTA-uniform)
      route_one_token(A.E, A.k, own_e, A.sel.offsets, A.sel.row_token, A.sel.row_slot, A.sel.slot_row, A.plan);
    __syncthreads();
    ctab = s_ctab;
    C = A.k;
  } else {
    ctab = plan_ctab(A.plan, A.E);
    const int C0 = A.plan[1];
    C = (C0 > 0 && C0 <= A.rows_max / kRows + A.E) ? C0 : 0;
  }
  const int fbs_g = A.pass[0].N / kMW, fbs_d = A.pass[1].N / kMW;
  const int items_g = C * fbs_g;
  const int items = items_g + C * fbs_d;
  const int glu_target = 4 * fbs_g;  // epilogue-warp arrivals that complete a chunk

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
    it.f0 = fb * kMW;
    return ok;
  };
  // stages of an item: a GLU item's alternate gate (even) and up (odd) over the same K range
  auto stages_of = [&](bool glu) -> int {
    const WmPass& W = A.pass[glu ? 0 : 1];
    return (glu ? 2 : 1) * (W.K / (128 * W.cps));
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
      const uint64_t stream_policy = l2_evict_first();
      while (ok) {
        const int u = next < items ? next : -1;
        if (!mbar_wait_bounded(&qempty[qs], qph ^ 1, abort_flag, A.err)) break;
        qitem[qs] = u;
        mbar_arrive(&qfull[qs]);
        if (++qs == kQ) { qs = 0; qph ^= 1; }
        if (u < 0) break;
        Item it;
        if (!item_of(u, it)) atomicOr(A.err, kErrIndex);
        next = atomicAdd(A.item_counter, 1);
        const WmPass& W = A.pass[it.glu ? 0 : 1];
        const int wrow = it.e * W.N + it.f0, cps = W.cps;
        const int nst = stages_of(it.glu);
        const uint32_t wbytes = (uint32_t)(kChunkA / 2 * cps) + (W.p0 ? 512u * cps : 0u),
                       abytes = it.glu ? 0u : (uint32_t)(kChunkB * cps);
        const size_t pblk = (size_t)(wrow / kMW) * (W.K / 128);  // the item's first staging block
        // a down item's weight tiles for the first stages go out before its chunk is complete;
        // its activation tiles (the chunk's GLU output) after
        const int npre = it.glu ? 0 : (nst < kStages ? nst : kStages);
        const int s_pre = s;
        for (int kc = 0; kc < nst; ++kc) {
          if (kc == npre && npre > 0) {
            if (!wait_chunk(A.chunk_done + it.c, glu_target, abort_flag, A.err)) { ok = false; break; }
            for (int j = 0; j < npre; ++j) {
              const int sj = (s_pre + j) % kStages;
              tma_load_3d(sB + sj * kBTile, &W.ta, 0, P * it.r0, j * cps, &full[sj]);
            }
          }
          if (!mbar_wait_bounded(&empty[s], ph ^ 1, abort_flag, A.err)) { ok = false; break; }
          mbar_arrive_expect_tx(&full[s], wbytes + abytes);
          const int kr = it.glu ? kc >> 1 : kc;  // K range of the stage
          tma_load_3d_stream(sA + s * kATile, (it.glu && (kc & 1)) ? &W.tw1 : &W.tw0, 0, wrow, kr * cps, &full[s],
                             stream_policy);
          if (W.p0)
            bulk_g2s_stream(stg + s * kSfBytes,
                            ((it.glu && (kc & 1)) ? W.p1 : W.p0) + (pblk + (size_t)kr * cps) * 512, 512u * cps,
                            &full[s], stream_policy);
          if (!it.glu && kc >= npre) tma_load_3d(sB + s * kBTile, &W.ta, 0, P * it.r0, kr * cps, &full[s]);
          if (++s == kStages) { s = 0; ph ^= 1; }
        }
        if (ok && npre == nst && npre > 0) {  // every stage went out before the wait
          if (!wait_chunk(A.chunk_done + it.c, glu_target, abort_flag, A.err)) break;
          for (int j = 0; j < npre; ++j) {
            const int sj = (s_pre + j) % kStages;
            tma_load_3d(sB + sj * kBTile, &W.ta, 0, P * it.r0, j * cps, &full[sj]);
          }
        }
      }
    }
  } else if (warp == 2 || warp == 3) {  // ---------------- scale and activation gather
    // Per stage: the weight rows' scales (gl = 0..63 takes rows gl and gl + 64, K-blocks 0-3 into
    // the first SFA block and 4-7 into the second); lanes 0..15 of warp 3 the activation rows'
    // scales (SFB); for GLU items the chunk's activation rows, 16-byte units (gl + 64 h) of the
    // 128-byte swizzled rows the MMA reads (unit j of row m at j ^ (m & 7)); rows past the chunk
    // are left out.
    const int gl = lane + (warp == 2 ? 0 : 32);
    const bool sfb_lane = warp == 3 && lane < RB;
    int s = 0, qs = 0;
    uint32_t ph = 0, qph = 0;
    bool ok = true;
    while (ok) {
      const int u = queue_pop(qfull, qempty, qitem, qs, qph, abort_flag, A.err);
      if (u < 0) break;
      Item it;
      item_of(u, it);
      const WmPass& W = A.pass[it.glu ? 0 : 1];
      const int srow = W.K / 32, spb = exp_pitch(W.K), cps = W.cps;
      const int nst = stages_of(it.glu);
      const size_t wrow = (size_t)it.e * W.N + it.f0;
      // token of a sorted row (checked: a bad one reads token 0 and sets the error word)
      auto token = [&](int r) -> size_t {
        if (A.ntok == 1) return 0;  // (one token: every row is its; the table may still be written)
        const int t = __ldg(A.row_token + r);
        if (t >= 0 && t < A.ntok) return (size_t)t;
        atomicOr(A.err, kErrIndex);
        return 0;
      };
      const bool act = sfb_lane && lane < P * it.nr;
      const size_t arow = !act ? 0 : it.glu ? token(it.r0 + lane / P) * P + lane % P : (size_t)P * it.r0 + lane;
      const uint8_t* as = W.sb + arow * spb;
      // GLU activation units gl + 64 h: chunk ch = unit / (8 RB) (of this stage's cps), row m, column j
      constexpr int kUnits = RB / 4;  // per gathering lane: 2 chunks x RB rows x 8 units over 64 lanes
      const uint8_t* asrc[kUnits];
      uint32_t adst[kUnits];
      bool aon[kUnits];
#pragma unroll
      for (int h = 0; h < kUnits; ++h) {
        const int unit = gl + 64 * h, ch = unit / (8 * RB), m = (unit >> 3) % RB, j = unit & 7;
        aon[h] = it.glu && ch < cps && m < P * it.nr;
        const size_t tr = aon[h] ? token(it.r0 + m / P) * P + m % P : 0;
        asrc[h] = W.sa + tr * W.K + 128 * ch + 16 * j;
        adst[h] = smem_u32(sB) + (uint32_t)(ch * kChunkB + m * 128 + ((j ^ (m & 7)) << 4));
      }
      const int npre = it.glu ? 0 : (nst < kStages ? nst : kStages);
      const int s_pre = s;
      for (int kc = 0; kc < nst; ++kc) {
        if (kc == npre && npre > 0) {  // a down item: its chunk's activation scales, for the stages issued so far
          int good = 1;
          if (warp == 3) {
            if (lane == 0) good = wait_chunk(A.chunk_done + it.c, glu_target, abort_flag, A.err) ? 1 : 0;
            good = __shfl_sync(0xffffffffu, good, 0);
          }
          if (!good) { ok = false; break; }
          if (sfb_lane)
            for (int j = 0; j < npre; ++j) {
              const int sj = (s_pre + j) % kStages;
              const uint32_t so = smem_u32(stg) + (uint32_t)(sj * kSfBytes) + 1024u + lane * 16;
              if (act)
                for (int c = 0; c < cps; ++c) cp_async4(so + 512 * c, as + 4 * (j * cps + c));
              cp_async_arrive(&full[sj]);
            }
        }
        if (!mbar_wait_warp(&empty[s], ph ^ 1, abort_flag, A.err)) { ok = false; break; }
        const int kr = it.glu ? kc >> 1 : kc;
        const uint32_t sbase = smem_u32(stg) + (uint32_t)(s * kSfBytes);
        // GLU: the activation rows of this K range (both the gate and the up stage copy them)
#pragma unroll
        for (int h = 0; h < kUnits; ++h)
          if (aon[h]) cp_async16(adst[h] + (uint32_t)(s * kBTile), asrc[h] + (size_t)kr * 128 * cps);
        // weight scales, unless the loading thread copies them: rows gl and gl + 64 of the item
        // (gate rows on even GLU stages, up rows on odd)
        const uint8_t* sw = (it.glu && (kc & 1)) ? W.s1 : W.s0;
#pragma unroll
        for (int rr = 0; rr < (W.p0 ? 0 : 2); ++rr) {
          const int r = gl + 64 * rr;
          const uint32_t so = sbase + (uint32_t)((r & 31) * 16 + (r >> 5) * 4);
          const uint8_t* src = sw + (wrow + r) * srow + 4 * kr * cps;
          for (int c = 0; c < cps; ++c) cp_async4(so + 512 * c, src + 4 * c);
        }
        if (sfb_lane) {
          if (kc >= npre) {
            if (act)
              for (int c = 0; c < cps; ++c) cp_async4(sbase + 1024u + lane * 16 + 512 * c, as + 4 * (kr * cps + c));
            cp_async_arrive(&full[s]);
          }
        } else {
          cp_async_arrive(&full[s]);
        }
        if (++s == kStages) { s = 0; ph ^= 1; }
      }
      if (ok && npre == nst && npre > 0) {  // every stage was gathered before the wait
        int good = 1;
        if (warp == 3) {
          if (lane == 0) good = wait_chunk(A.chunk_done + it.c, glu_target, abort_flag, A.err) ? 1 : 0;
          good = __shfl_sync(0xffffffffu, good, 0);
        }
        if (!good) break;
        if (sfb_lane)
          for (int j = 0; j < npre; ++j) {
            const int sj = (s_pre + j) % kStages;
            const uint32_t so = smem_u32(stg) + (uint32_t)(sj * kSfBytes) + 1024u + lane * 16;
            if (act)
              for (int c = 0; c < cps; ++c) cp_async4(so + 512 * c, as + 4 * (j * cps + c));
            cp_async_arrive(&full[sj]);
          }
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");  // nothing lands after the block has gone
  } else if (warp == 1) {  // ---------------- MMA issue (converged warp, one elected lane)
    int s = 0, qs = 0, n = 0;
    uint32_t ph = 0;
    uint32_t qph = 0;
    bool ok = true;
    while (ok) {
      const int u = queue_pop(qfull, qempty, qitem, qs, qph, abort_flag, A.err);
      if (u < 0) break;
      const bool glu = u < items_g;
      const int cps = A.pass[glu ? 0 : 1].cps;
      const int nst = stages_of(glu);
      const int b = n & 1;
      const uint32_t acc = tmem + b * kAccCols;
      if (!mbar_wait_warp(&acce[b], (uint32_t)(((n >> 1) & 1) ^ 1), abort_flag, A.err)) { ok = false; break; }
      tc_fence_after();
      for (int kc = 0; kc < nst; ++kc) {
        if (!mbar_wait_warp(&full[s], ph, abort_flag, A.err)) { ok = false; break; }
        const uint32_t tsf = tmem + kSfCol + 16 * s;
        const uint32_t st0 = smem_u32(stg + s * kSfBytes);
        const uint32_t a0 = smem_u32(sA + s * kATile), b0 = smem_u32(sB + s * kBTile);
        const uint32_t d = acc + ((glu && (kc & 1)) ? 16u : 0u);
        const int kfirst = glu ? (kc >> 1) : kc;  // K range index: accumulate from the second on
        if (elect_one()) {
          fence_async_smem();  // the scales and activation rows arrived through cp.async
          tc_fence_after();
          for (int c = 0; c < cps; ++c) {
            asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(tsf + 4 * c),
                         "l"(sdesc_sf(st0 + 512 * c)));
            asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(tsf + 8 + 4 * c),
                         "l"(sdesc_sf(st0 + 1024 + 512 * c)));
          }
          for (int kk = 0; kk < 4 * cps; ++kk) {
            const int c = kk >> 2, q = kk & 3;
            umma_mx(d, sdesc_sw128(a0 + c * kChunkA + q * 32), sdesc_sw128(b0 + c * kChunkB + q * 32), idesc_wm(q),
                    tsf + 4 * c, tsf + 8 + 4 * c, (kfirst | kk) != 0 ? 1u : 0u);
          }
          umma_commit(&empty[s]);
        }
        __syncwarp();
        if (++s == kStages) { s = 0; ph ^= 1; }
      }
      if (!ok) break;
      if (elect_one()) umma_commit(&accf[b]);
      __syncwarp();
      ++n;
    }
    if (elect_one()) {  // every issued MMA has completed before the tensor memory is released
      umma_commit(drain);
      volatile int no_abort = 0;
      mbar_wait_bounded(drain, 0, &no_abort, A.err);
    }
    __syncwarp();
  } else {  // ---------------- epilogue, warps 4..7: tensor-memory lanes 32q..32q+31
    // Accumulator lane = weight row (32q + lane) of the item; column m = activation row m (sorted
    // row m / P, part m % P).
    const int q = warp - kEpiWarp0;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
    int qs = 0, n = 0;
    uint32_t qph = 0;
    for (;;) {
      const int u = queue_pop(qfull, qempty, qitem, qs, qph, abort_flag, A.err);
      if (u < 0) break;
      Item it;
      item_of(u, it);
      const int b = n & 1;
      if (!mbar_wait_warp(&accf[b], (uint32_t)((n >> 1) & 1), abort_flag, A.err)) break;
      ++n;
      tc_fence_after();
      uint32_t g[16], v[16];
      tmem_ld16(lane_base + b * kAccCols, g);
      if (it.glu) tmem_ld16(lane_base + b * kAccCols + 16, v);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acce[b]);  // the accumulator may be overwritten now
      const int f = it.f0 + 32 * q + lane;      // this thread's weight row (output feature)
      if (it.glu) {
        const int N = A.pass[0].N, spo = exp_pitch(N);
#pragma unroll
        for (int j = 0; j < kRows; ++j) {
          if (j >= it.nr) break;  // warp-uniform
          float gv = __uint_as_float(g[P * j]), uv = __uint_as_float(v[P * j]);
          if (P == 2) {
            gv += __uint_as_float(g[2 * j + 1]);
            uv += __uint_as_float(v[2 * j + 1]);
          }
          // silu(g) = g / (1 + e^-g), fast forms (~1e-6 relative)
          const float a = bf16_to_f32(f32_to_bf16(__fdividef(gv, 1.0f + __expf(-gv)) * uv));
          const size_t brow = (size_t)P * (it.r0 + j);
          // the 32 features of this warp are one scale block
          if (P == 1) {
            const int X = mxfp8_block_exp(warp_max(fabsf(a)));
            A.aq[brow * N + f] = (uint8_t)e4m3_code(a, X);
            if (lane == 0) A.aqs[brow * spo + f / 32] = (uint8_t)(X + 127);
          } else {  // hi, then the exact remainder on its own block exponent
            const int X0 = split_block_exp(warp_max(fabsf(a)));
            const uint32_t c0 = e4m3_code(a, X0);
            const float rem = a - mul_pow2(e4m3x2_value(c0).x, X0);
            const int X1 = split_block_exp(warp_max(fabsf(rem)));
            A.aq[brow * N + f] = (uint8_t)c0;
            A.aq[(brow + 1) * N + f] = (uint8_t)e4m3_code(rem, X1);
            if (lane == 0) {
              A.aqs[brow * spo + f / 32] = (uint8_t)(X0 + 127);
              A.aqs[(brow + 1) * spo + f / 32] = (uint8_t)(X1 + 127);
            }
          }
        }
        // publish this warp's part of the chunk's GLU output (release)
        __syncwarp();
        if (lane == 0) {
          asm volatile("fence.proxy.async.global;" ::: "memory");
          __threadfence();
          atomicAdd(A.chunk_done + it.c, 1);
        }
      } else {
        const int L = A.pass[1].N;
#pragma unroll
        for (int j = 0; j < kRows; ++j) {
          if (j >= it.nr) break;
          float o = __uint_as_float(g[P * j]);
          if (P == 2) o += __uint_as_float(g[2 * j + 1]);
          A.o_out[(size_t)(it.r0 + j) * L + f] = o;
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

static_assert(kATile % 1024 == 0, "128-byte swizzle alignment");

template <int P, int RB>
cudaError_t launch_t(UWmArgs& a, int items_max, cudaStream_t s) {
  constexpr size_t kSmem = WmShape<RB>::kSmem;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(umma_wm_kernel<P, RB>), kSmem);
  if (e != cudaSuccess) return e;
  int grid = num_sms();  // one CTA per SM (the shared memory allows no second)
  if (items_max < grid) grid = items_max > 0 ? items_max : 1;
  return launch_pdl(umma_wm_kernel<P, RB>, dim3(grid), dim3(kThreads), kSmem, s, a);
}

// dst = src's scales [rows][K/32] in the staging image: block (rb, c) of 512 bytes holds, at
// lane l, word w, the four scales of row 128 rb + 32 w + l for K-blocks 4c .. 4c + 3.
__global__ void pack_scales_kernel(const uint32_t* __restrict__ src, long long words, int kc, uint32_t* dst) {
  for (long long o = blockIdx.x * (long long)blockDim.x + threadIdx.x; o < words; o += (long long)gridDim.x * blockDim.x) {
    const long long blk = o >> 7;
    const int l = (int)(o >> 2) & 31, w = (int)o & 3;
    const long long rb = blk / kc;
    const int c = (int)(blk - rb * kc);
    dst[o] = src[(rb * kMW + 32 * w + l) * kc + c];
  }
}

// The same image for the many-token GLU tile of 64 gate rows and their 64 up rows: block (fb, c)
// holds, at lane l, word w, the four scales of tile row 32 w + l (gate row 64 fb + 32 w + l for
// w < 2, up row 64 fb + 32 (w - 2) + l otherwise) for K-blocks 4c .. 4c + 3.
__global__ void pack_scales_glu_kernel(const uint32_t* __restrict__ gate, const uint32_t* __restrict__ up,
                                       long long words, int kc, uint32_t* dst) {
  for (long long o = blockIdx.x * (long long)blockDim.x + threadIdx.x; o < words; o += (long long)gridDim.x * blockDim.x) {
    const long long blk = o >> 7;
    const int l = (int)(o >> 2) & 31, w = (int)o & 3;
    const long long fb = blk / kc;
    const int c = (int)(blk - fb * kc);
    dst[o] = (w < 2 ? gate : up)[(fb * 64 + 32 * (w & 1) + l) * kc + c];
  }
}

}  // namespace

cudaError_t launch_pack_scales_glu(const uint8_t* gate, const uint8_t* up, long long rows, int K, uint8_t* dst,
                                   cudaStream_t s) {
  if (rows % 64 || K % 128) return cudaErrorInvalidValue;
  const long long words = 2 * rows * (K / 128);
  const int grid = (int)((words + 255) / 256 < 4096 ? (words + 255) / 256 : 4096);
  pack_scales_glu_kernel<<<grid > 0 ? grid : 1, 256, 0, s>>>(reinterpret_cast<const uint32_t*>(gate),
                                                           reinterpret_cast<const uint32_t*>(up), words, K / 128,
                                                           reinterpret_cast<uint32_t*>(dst));
  return cudaGetLastError();
}

cudaError_t launch_pack_scales(const uint8_t* src, long long rows, int K, uint8_t* dst, cudaStream_t s) {
  if (rows % kMW || K % 128) return cudaErrorInvalidValue;
  const long long words = rows * (K / 128);
  const int grid = (int)((words + 255) / 256 < 4096 ? (words + 255) / 256 : 4096);
  pack_scales_kernel<<<grid > 0 ? grid : 1, 256, 0, s>>>(reinterpret_cast<const uint32_t*>(src), words, K / 128,
                                                       reinterpret_cast<uint32_t*>(dst));
  return cudaGetLastError();
}

cudaError_t launch_umma_decode(const k3moe_dims& d, const k3moe_weights& w, const PackedScales* ps, int32_t* plan,
                               const uint8_t* zq, const uint8_t* zqs, const int32_t* row_token, int P, int T,
                               uint8_t* aq, uint8_t* aqs, float* o_rows, int* chunk_done, uint32_t* err,
                               cudaStream_t s, const DecodeSelect* sel) {
  if (d.latent % 128 || d.inter % 128 || (P != 1 && P != 2)) return cudaErrorInvalidValue;
  if (sel && (T != 1 || d.top_k > 32)) return cudaErrorInvalidValue;
  // activation rows per chunk: P x (sorted rows of one expert, at most T and kRows)
  const int RB = P * (T < kRows ? T : kRows) <= 8 ? 8 : 16;
  UWmArgs A{};
  const int rows = T * d.top_k;
  WmPass& G = A.pass[0];
  G.cps = d.latent % 256 == 0 ? 2 : 1;
  const uint64_t wrows = (uint64_t)d.n_experts * d.inter;
  if (!make_tmap_fp4_chunks(&G.tw0, w.gate_q, d.latent, wrows, (uint64_t)d.latent / 2, kMW, (uint32_t)G.cps) ||
      !make_tmap_fp4_chunks(&G.tw1, w.up_q, d.latent, wrows, (uint64_t)d.latent / 2, kMW, (uint32_t)G.cps))
    return cudaErrorInvalidValue;
  G.s0 = w.gate_s; G.s1 = w.up_s; G.sa = zq; G.sb = zqs;
  if (ps) { G.p0 = ps->gate; G.p1 = ps->up; }
  G.N = d.inter; G.K = d.latent;
  WmPass& D = A.pass[1];
  D.cps = d.inter % 256 == 0 ? 2 : 1;
  if (!make_tmap_fp4_chunks(&D.tw0, w.down_q, d.inter, (uint64_t)d.n_experts * d.latent, (uint64_t)d.inter / 2, kMW,
                            (uint32_t)D.cps) ||
      !make_tmap_3d_chunks(&D.ta, aq, 1, 128, (uint64_t)P * rows, (uint64_t)d.inter, (uint64_t)d.inter / 128,
                           (uint32_t)RB, (uint32_t)D.cps, true))
    return cudaErrorInvalidValue;
  D.s0 = w.down_s; D.sb = aqs;
  if (ps) D.p0 = ps->down;
  D.N = d.latent; D.K = d.inter;
  const int chunks = rows / kRows + d.n_experts;
  const int items_max = chunks * (d.inter / kMW + d.latent / kMW);
  A.plan = plan; A.row_token = row_token; A.ntok = T; A.E = d.n_experts; A.rows_max = rows;
  A.aq = aq; A.aqs = aqs; A.o_out = o_rows; A.chunk_done = chunk_done; A.err = err;
  A.item_counter = chunk_done + plan_chunks_max(d, T);
  if (sel) A.sel = *sel;
  A.k = d.top_k;
  if (P == 1) return launch_t<1, 8>(A, items_max, s);
  return RB == 8 ? launch_t<2, 8>(A, items_max, s) : launch_t<2, 16>(A, items_max, s);
}

}  // namespace k3moe
