// Routing building blocks shared by the routing kernels and the decode expert kernel (which,
// for one token, selects the experts itself): the top-k selection of one token by one CTA of
// 256 threads, and the permutation and plan of one token's selection.
//
// "kimi-k3-mlx", Architecture table: each token activates 16 of 896 routed experts.
// Selection keeps the k largest logits; equal logits go to the lower expert index (NaN ranks
// below every number, -0 equals +0). The kept indices are written in ascending order and their
// weights are the softmax over the kept logits, which equals softmax over all logits
// renormalised over the kept ones.
#pragma once

#include "k3moe_device.cuh"
#include "k3moe_internal.cuh"

namespace k3moe {
namespace {

constexpr int kMaxE = 1024;

// Order-preserving 32-bit key of a logit: larger logit -> larger key. -0 equals +0; NaN gets
// 1, below every number (numbers map to >= 0x007fffff); 0 marks an empty or taken slot.
__device__ __forceinline__ uint32_t sort_key(float v) {
  uint32_t u = __float_as_uint(v);
  if (v == 0.0f) u = 0u;
  if (v != v) return 1u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// One CTA of 256 threads routes one token. Radix select over the 32-bit keys, one 8-bit digit
// per pass (a shared histogram, then one warp finds the digit holding the k-th largest key),
// gives the k-th largest key; keys above it are kept, and of the keys equal to it the
// lowest-indexed ones (ranked by a block count in index order). One warp sorts the kept
// experts by index and writes them with the softmax weights over their logits.
constexpr int kTopkThreads = 256;
constexpr int kTopkKeys = kMaxE / kTopkThreads;  // keys per thread
// Returns, to thread lane < k of warp 0, the expert it wrote to slot lane (-1 elsewhere).
// store = false: nothing is written.
__device__ int block_topk(const float* __restrict__ logits, int t, int E, int k, int32_t* idx, float* w,
                          bool store = true) {
  __shared__ int hist[256];
  __shared__ int s_digit, s_above, s_nsel, s_full;
  __shared__ int wcnt[kTopkKeys][kTopkThreads / 32];
  __shared__ int sel_e[32];
  __shared__ float sel_l[32];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const unsigned lt = (1u << lane) - 1u;
  const float* lg = logits + (size_t)t * E;
  uint32_t key[kTopkKeys];
#pragma unroll
  for (int i = 0; i < kTopkKeys; ++i) {
    const int e = tid + kTopkThreads * i;
    key[i] = e < E ? sort_key(lg[e]) : 0u;  // 0 = no expert (below every key, even NaN's)
  }
  if (tid == 0) s_nsel = 0;
  uint32_t thr = 0u, pmask = 0u;
  int need = k;
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    hist[tid] = 0;
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kTopkKeys; ++i)
      if (key[i] != 0u && (key[i] & pmask) == thr) atomicAdd(&hist[(key[i] >> shift) & 255], 1);
    __syncthreads();
    if (wid == 0) {  // digits in descending order: lane l covers 255 - 8l .. 248 - 8l
      int c[8], sum = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = hist[255 - 8 * lane - j];
        sum += c[j];
      }
      int inc = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
      }
      int run = inc - sum;
      if (run < need && need <= inc) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (run < need && need <= run + c[j]) {
            s_digit = 255 - 8 * lane - j;
            s_above = run;
            s_full = c[j] == need - run;  // the bucket holds exactly the keys still needed
          }
          run += c[j];
        }
      }
    }
    __syncthreads();
    thr |= (uint32_t)s_digit << shift;
    pmask |= 255u << shift;
    need -= s_above;
    if (s_full) break;  // every key with this prefix is selected: the lower digits decide nothing
  }
  // Keys compare on their top bytes kept so far (pmask): above thr are selected; equal to thr
  // (the boundary; the k-th largest key itself when all four digits ran) take `need` of them,
  // lowest index first
  int rank_in_warp[kTopkKeys];
#pragma unroll
  for (int i = 0; i < kTopkKeys; ++i) {
    const unsigned b = __ballot_sync(0xffffffffu, key[i] != 0u && (key[i] & pmask) == thr);
    rank_in_warp[i] = __popc(b & lt);
    if (lane == 0) wcnt[i][wid] = __popc(b);
  }
  __syncthreads();
  int before = 0;
#pragma unroll
  for (int i = 0; i < kTopkKeys; ++i) {
    int bw = 0, tot = 0;
#pragma unroll
    for (int x = 0; x < kTopkThreads / 32; ++x) {
      bw += x < wid ? wcnt[i][x] : 0;
      tot += wcnt[i][x];
    }
    const uint32_t km = key[i] & pmask;
    const bool sel = key[i] != 0u && (km > thr || (km == thr && before + bw + rank_in_warp[i] < need));
    if (sel) {
      const int slot = atomicAdd(&s_nsel, 1);
      const int e = tid + kTopkThreads * i;
      sel_e[slot] = e;
      sel_l[slot] = lg[e];
    }
    before += tot;
  }
  __syncthreads();
  if (wid == 0) {
    int e = lane < k ? sel_e[lane] : 0x7fffffff;
    float l = lane < k ? sel_l[lane] : 0.f;
    // bitonic sort by expert index, ascending
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        const int pe = __shfl_xor_sync(0xffffffffu, e, stride);
        const float pl = __shfl_xor_sync(0xffffffffu, l, stride);
        const bool up = (lane & size) == 0 || size == 32;
        const bool lower = (lane & stride) == 0;
        if (lower == up ? pe < e : pe > e) {
          e = pe;
          l = pl;
        }
      }
    }
    float lmax = lane < k ? l : -3.402823466e38f;
    lmax = warp_max(lmax);
    const float ex = lane < k ? expf(l - lmax) : 0.f;
    float sum = ex;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (store && lane < k) {
      idx[(size_t)t * k + lane] = e;
      w[(size_t)t * k + lane] = ex / sum;
    }
    return lane < k ? e : -1;
  }
  return -1;
}

// One token, k distinct valid experts held in ascending order by threads 0..k-1 (own_e): slot j
// is sorted row j, each expert one run of one row and one chunk. The same outputs as
// block_route_tiny gives for this case, in a few short loops.
__device__ void route_one_token(int E, int k, int own_e, int32_t* offsets, int32_t* row_token, int32_t* row_slot,
                                int32_t* slot_row, int32_t* plan) {
  __shared__ int s_sel[32];
  const int tid = threadIdx.x;
  if (tid < k) s_sel[tid] = own_e;
  __syncthreads();
  for (int e = tid; e <= E; e += blockDim.x) {  // rows of the experts below e
    int c = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) c += (j < k && s_sel[j] < e) ? 1 : 0;  // independent loads
    offsets[e] = c;
  }
  if (tid < k) {
    const int4 run = make_int4(own_e, tid, 1, 0);
    row_token[tid] = 0;
    row_slot[tid] = tid;
    slot_row[tid] = tid;
    plan[2 + tid] = own_e;
    plan[2 + E + tid] = tid;
    plan_ctab(plan, E)[tid] = run;
    plan_ctab64(plan, E, k)[1 + tid] = run;
  }
  if (tid == 0) {
    plan[0] = k;
    plan[1] = k;
    plan[2 + E + k] = k;
    plan_ctab64(plan, E, k)[0] = make_int4(k, 0, 0, 0);
  }
}

}  // namespace
}  // namespace k3moe
