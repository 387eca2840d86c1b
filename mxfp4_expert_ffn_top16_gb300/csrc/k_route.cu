// Routing: top-k selection with renormalised weights, the token-by-expert permutation, and
// the schedule ("plan") the expert kernels read.
//
// "kimi-k3-mlx", Architecture table: each token activates 16 of 896 routed experts.
// Selection keeps the k largest logits; equal logits go to the lower expert index (NaN
// ranks below every number, -0 equals +0). The kept indices are written in ascending order
// and their weights are the softmax over the kept logits, which equals softmax over all
// logits renormalised over the kept ones.
//
// Top-k: one warp per token, each lane holding E/32 logits as order-preserving 64-bit keys
// (float key, then inverted index) in registers; k rounds of a warp max.
// Permutation: rows grouped by expert, token order inside an expert (the order a stable
// counting sort gives). Histogram -> exclusive scan -> scatter; the scatter walks tokens in
// chunks of 32 (one per lane) and ranks a (token, expert) pair inside its chunk with a
// per-expert lane bitmask, so the result is exact and deterministic.
#include "k3moe_device.cuh"
#include "k3moe_internal.cuh"

namespace k3moe {
namespace {

constexpr int kMaxE = 1024;
constexpr int kMaxPerLane = kMaxE / 32;

// Order-preserving 32-bit key of a logit: larger logit -> larger key. -0 equals +0; NaN gets
// 1, below every number (numbers map to >= 0x007fffff); 0 marks an empty or taken slot.
__device__ __forceinline__ uint32_t sort_key(float v) {
  uint32_t u = __float_as_uint(v);
  if (v == 0.0f) u = 0u;
  if (v != v) return 1u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w > v ? w : v;
  }
  return v;
}

// One warp selects the top-k of one token's logits row. Lanes j < k end with
// (*sel_idx, *sel_logit) = the j-th largest; returns nothing for lanes >= k.
__device__ void warp_topk(const float* __restrict__ lg, int E, int k, int lane, int* sel_idx,
                          float* sel_logit) {
  // slot j of this lane holds expert lane + 32 j; within a lane the lowest j wins ties
  uint32_t keys[kMaxPerLane];
  const int per = (E + 31) / 32;
#pragma unroll
  for (int j = 0; j < kMaxPerLane; ++j) {
    const int e = lane + 32 * j;
    keys[j] = (j < per && e < E) ? sort_key(lg[e]) : 0u;
  }
  // (key, inverted expert index) of this lane's best remaining slot
  auto local_best = [&]() -> unsigned long long {
    uint32_t bk = 0u;
    int bj = 0;
#pragma unroll
    for (int j = 0; j < kMaxPerLane; ++j)
      if (keys[j] > bk) { bk = keys[j]; bj = j; }
    return bk == 0u ? 0ull
                    : ((unsigned long long)bk << 32) | (uint32_t)(0xffffffffu - (uint32_t)(lane + 32 * bj));
  };
  unsigned long long best = local_best();
  int my_idx = -1;
  for (int r = 0; r < k; ++r) {
    const unsigned long long win = warp_max_u64(best);
    const int widx = (int)(0xffffffffu - (uint32_t)(win & 0xffffffffu));
    if (lane == r) my_idx = widx;
    if ((widx & 31) == lane) {  // owner takes the slot and rescans
      const int wj = widx >> 5;
#pragma unroll
      for (int j = 0; j < kMaxPerLane; ++j)
        if (j == wj) keys[j] = 0u;
      best = local_best();
    }
  }
  *sel_idx = my_idx;
  *sel_logit = (lane < k && my_idx >= 0) ? lg[my_idx] : 0.0f;
}

// Writes one token's k indices in ascending order with their renormalised weights.
__device__ void warp_write_topk(int sel, float l, int k, int lane, int32_t* idx_row, float* w_row,
                                int* smem_idx_row) {
  const bool act = lane < k;
  const float lmax = __shfl_sync(0xffffffffu, l, 0);  // lane 0 holds the largest
  const float ex = act ? expf(l - lmax) : 0.0f;
  float sum = ex;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  int rank = 0;
  for (int j = 0; j < k; ++j) {
    const int other = __shfl_sync(0xffffffffu, sel, j);
    rank += (act && other < sel) ? 1 : 0;
  }
  if (act) {
    idx_row[rank] = sel;
    w_row[rank] = ex / sum;
    if (smem_idx_row) smem_idx_row[rank] = sel;
  }
}

__global__ void topk_kernel(const float* __restrict__ logits, int T, int E, int k, int32_t* idx,
                            float* w) {
  const int lane = threadIdx.x & 31;
  const int tok = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (tok >= T) return;
  int sel;
  float l;
  warp_topk(logits + (size_t)tok * E, E, k, lane, &sel, &l);
  warp_write_topk(sel, l, k, lane, idx + (size_t)tok * k, w + (size_t)tok * k, nullptr);
}

// ---------------------------------------------------------------- block-level building blocks
// Exclusive scan of cnt[0..n) in shared memory (n <= blockDim.x, blockDim.x a multiple of 32);
// returns the total. Warp shuffles within each warp, one warp over the warp totals: three
// block barriers in all.
__device__ int block_excl_scan(int* cnt, int n, int* tmp) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nw = blockDim.x >> 5;
  const int v = tid < n ? cnt[tid] : 0;
  int x = v;  // inclusive scan within the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) tmp[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int w = lane < nw ? tmp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    tmp[lane] = w;  // inclusive totals of warps 0..lane
  }
  __syncthreads();
  const int total = tmp[nw - 1];
  if (tid < n) cnt[tid] = (wid > 0 ? tmp[wid - 1] : 0) + x - v;
  __syncthreads();
  return total;
}

// Plan from offsets[E+1] held in shared memory: active experts, chunk prefix, the chunk
// table ctab[c] = {expert, first sorted row, rows (<= 8), 0} in expert order, and the table of
// chunks of up to kUmmaChunkRows rows for the tensor-core expert GEMM. rows_max = T * k fixes
// where the second table sits.
__device__ void build_plan(const int* off, int E, int rows_max, int32_t* plan, int* tmp, int* flag,
                           int* chunks) {
  const int tid = threadIdx.x;
  int4* ctab = plan_ctab(plan, E);
  int4* ctab64 = plan_ctab64(plan, E, rows_max);
  const int m = tid < E ? off[tid + 1] - off[tid] : 0;
  if (tid < E) {
    flag[tid] = m > 0 ? 1 : 0;
    chunks[tid] = (m + kGemvTokens - 1) / kGemvTokens;
  }
  __syncthreads();
  const int D = block_excl_scan(flag, E, tmp);
  const int C = block_excl_scan(chunks, E, tmp);
  if (tid < E && m > 0) {
    plan[2 + flag[tid]] = tid;
    plan[2 + E + flag[tid]] = chunks[tid];
    for (int q = 0; q * kGemvTokens < m; ++q)
      ctab[chunks[tid] + q] = make_int4(tid, off[tid] + q * kGemvTokens, min(kGemvTokens, m - q * kGemvTokens), 0);
  }
  if (tid == 0) {
    plan[0] = D;
    plan[1] = C;
    plan[2 + E + D] = C;
  }
  __syncthreads();
  if (tid < E) flag[tid] = (m + kUmmaChunkRows - 1) / kUmmaChunkRows;
  __syncthreads();
  const int C64 = block_excl_scan(flag, E, tmp);
  if (tid < E)
    for (int q = 0; q * kUmmaChunkRows < m; ++q)
      ctab64[1 + flag[tid] + q] =
          make_int4(tid, off[tid] + q * kUmmaChunkRows, min(kUmmaChunkRows, m - q * kUmmaChunkRows), 0);
  if (tid == 0) ctab64[0] = make_int4(C64, 0, 0, 0);
}

// Scatter of tokens [t0, t1) by one warp, given base[e] = first free row of each expert.
__device__ void warp_scatter(const int32_t* __restrict__ idx, int t0, int t1, int E, int k,
                             int* base, unsigned* mask, int32_t* row_token, int32_t* row_slot,
                             int32_t* slot_row, uint32_t* err) {
  const int lane = threadIdx.x & 31;
  const unsigned lt = (1u << lane) - 1u;
  for (int c0 = t0; c0 < t1; c0 += 32) {
    const int t = c0 + lane;
    const bool v = t < t1;
    for (int j = 0; j < k; ++j) {
      const int e = v ? idx[(size_t)t * k + j] : -1;
      if (v && (e < 0 || e >= E)) atomicOr(err, kErrIndex);
      if (v && e >= 0 && e < E) atomicOr(&mask[e], 1u << lane);
    }
    __syncwarp();
    for (int j = 0; j < k; ++j) {
      const int e = v ? idx[(size_t)t * k + j] : -1;
      if (v && e >= 0 && e < E) {
        const int r = base[e] + __popc(mask[e] & lt);
        row_token[r] = t;
        row_slot[r] = j;
        slot_row[(size_t)t * k + j] = r;
      }
    }
    __syncwarp();
    for (int j = 0; j < k; ++j) {
      const int e = v ? idx[(size_t)t * k + j] : -1;
      if (v && e >= 0 && e < E) {
        const unsigned m = mask[e];
        if ((m & lt) == 0u) {  // lowest lane holding e advances its base and clears
          base[e] += __popc(m);
          mask[e] = 0u;
        }
      }
    }
    __syncwarp();
  }
}

// ---------------------------------------------------------------- single-CTA permutation
// For T*k small: histogram, scan, scatter and plan in one block of 1024 threads.
// With `logits` given, the block first selects the top-k of each token (one warp per token)
// into idx / w, so decode routing is a single launch.
__global__ void __launch_bounds__(1024) permute_small_kernel(const float* __restrict__ logits,
                                                             float* w, int32_t* idx, int T,
                                                             int E, int k, int32_t* offsets,
                                                             int32_t* row_token, int32_t* row_slot,
                                                             int32_t* slot_row, int32_t* plan,
                                                             uint32_t* err) {
  __shared__ int cnt[kMaxE + 1];
  __shared__ int tmp[1024];
  __shared__ int flag[kMaxE];
  __shared__ int chunks[kMaxE];
  __shared__ unsigned mask[kMaxE];
  const int tid = threadIdx.x;
  pdl_wait();
  pdl_trigger();
  if (logits) {
    const int lane = tid & 31;
    for (int t = tid >> 5; t < T; t += blockDim.x >> 5) {
      int sel;
      float l;
      warp_topk(logits + (size_t)t * E, E, k, lane, &sel, &l);
      warp_write_topk(sel, l, k, lane, idx + (size_t)t * k, w + (size_t)t * k, nullptr);
    }
    __syncthreads();
  }
  if (tid <= E) cnt[tid] = 0;
  if (tid < E) mask[tid] = 0u;
  __syncthreads();
  for (int i = tid; i < T * k; i += blockDim.x) {
    const int e = idx[i];
    if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);
  }
  __syncthreads();
  const int total = block_excl_scan(cnt, E, tmp);
  if (tid == 0) cnt[E] = total;
  __syncthreads();
  if (tid <= E) offsets[tid] = cnt[tid];
  __syncthreads();
  // plan reads the offsets before the scatter turns cnt into running bases
  build_plan(cnt, E, T * k, plan, tmp, flag, chunks);
  __syncthreads();
  if (tid < 32) warp_scatter(idx, 0, T, E, k, cnt, mask, row_token, row_slot, slot_row, err);
}

// ---------------------------------------------------------------- multi-CTA permutation
constexpr int kBlockTokens = 256;

__global__ void __launch_bounds__(256) hist_kernel(const int32_t* __restrict__ idx, int T, int E,
                                                   int k, int32_t* hist) {
  __shared__ int cnt[kMaxE];
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  const int t0 = blockIdx.x * kBlockTokens, t1 = min(T, t0 + kBlockTokens);
  for (int i = t0 * k + threadIdx.x; i < t1 * k; i += blockDim.x) {
    const int e = idx[i];
    if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[(size_t)blockIdx.x * E + e] = cnt[e];
}

// One block of 1024 threads: per-expert running sums over token blocks -> offsets, then
// hist[b][e] becomes the first row of expert e for token block b; plan from offsets.
__global__ void __launch_bounds__(1024) scan_kernel(int32_t* hist, int nblk, int E, int rows_max,
                                                    int32_t* offsets, int32_t* plan) {
  __shared__ int cnt[kMaxE + 1];
  __shared__ int tmp[1024];
  __shared__ int flag[kMaxE];
  __shared__ int chunks[kMaxE];
  const int tid = threadIdx.x;
  int tot = 0;
  if (tid < E)
    for (int b = 0; b < nblk; ++b) tot += hist[(size_t)b * E + tid];
  if (tid < E) cnt[tid] = tot;
  __syncthreads();
  const int total = block_excl_scan(cnt, E, tmp);
  if (tid == 0) cnt[E] = total;
  __syncthreads();
  if (tid <= E) offsets[tid] = cnt[tid];
  if (tid < E) {
    int run = cnt[tid];
    for (int b = 0; b < nblk; ++b) {
      const int h = hist[(size_t)b * E + tid];
      hist[(size_t)b * E + tid] = run;
      run += h;
    }
  }
  __syncthreads();
  build_plan(cnt, E, rows_max, plan, tmp, flag, chunks);
}

__global__ void __launch_bounds__(32) scatter_kernel(const int32_t* __restrict__ idx, int T, int E,
                                                     int k, const int32_t* base_g,
                                                     int32_t* row_token, int32_t* row_slot,
                                                     int32_t* slot_row, uint32_t* err) {
  __shared__ int base[kMaxE];
  __shared__ unsigned mask[kMaxE];
  for (int e = threadIdx.x; e < E; e += 32) {
    base[e] = base_g[(size_t)blockIdx.x * E + e];
    mask[e] = 0u;
  }
  __syncwarp();
  const int t0 = blockIdx.x * kBlockTokens, t1 = min(T, t0 + kBlockTokens);
  warp_scatter(idx, t0, t1, E, k, base, mask, row_token, row_slot, slot_row, err);
}

// Plan from caller-supplied offsets. Offsets that are not a non-decreasing sequence from 0
// to at most rows_max set the index bit of the error word and give an empty plan.
__global__ void __launch_bounds__(1024) plan_kernel(const int32_t* __restrict__ offsets, int E,
                                                    int rows_max, int32_t* plan, uint32_t* err) {
  __shared__ int off[kMaxE + 1];
  __shared__ int tmp[1024];
  __shared__ int flag[kMaxE];
  __shared__ int chunks[kMaxE];
  __shared__ int bad;
  if (threadIdx.x == 0) bad = 0;
  __syncthreads();
  for (int e = threadIdx.x; e <= E; e += blockDim.x) {
    off[e] = offsets[e];
    if (off[e] < 0 || off[e] > rows_max) bad = 1;
  }
  __syncthreads();
  if (threadIdx.x < E && off[threadIdx.x + 1] < off[threadIdx.x]) bad = 1;
  if (threadIdx.x == 0 && off[0] != 0) bad = 1;
  __syncthreads();
  if (bad) {
    if (threadIdx.x == 0) {
      plan[0] = 0;
      plan[1] = 0;
      plan_ctab64(plan, E, rows_max)[0] = make_int4(0, 0, 0, 0);
      atomicOr(err, kErrIndex);
    }
    return;
  }
  build_plan(off, E, rows_max, plan, tmp, flag, chunks);
}

}  // namespace

cudaError_t launch_topk(const float* logits, int T, int E, int k, int32_t* idx, float* w,
                        cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  const int warps = 8;
  topk_kernel<<<(T + warps - 1) / warps, 32 * warps, 0, s>>>(logits, T, E, k, idx, w);
  return cudaGetLastError();
}

cudaError_t launch_permute(const int32_t* idx, int T, int E, int k, int32_t* offsets,
                           int32_t* row_token, int32_t* row_slot, int32_t* slot_row,
                           int32_t* plan, int32_t* scratch, uint32_t* err, cudaStream_t s) {
  if (T <= kBlockTokens) {
    permute_small_kernel<<<1, 1024, 0, s>>>(nullptr, nullptr, const_cast<int32_t*>(idx), T, E, k,
                                            offsets, row_token, row_slot, slot_row, plan, err);
    return cudaGetLastError();
  }
  const int nblk = (T + kBlockTokens - 1) / kBlockTokens;
  hist_kernel<<<nblk, 256, 0, s>>>(idx, T, E, k, scratch);
  scan_kernel<<<1, 1024, 0, s>>>(scratch, nblk, E, T * k, offsets, plan);
  scatter_kernel<<<nblk, 32, 0, s>>>(idx, T, E, k, scratch, row_token, row_slot, slot_row, err);
  return cudaGetLastError();
}

cudaError_t launch_route_tail_small(const float* logits, int T, int E, int k, int32_t* idx, float* w,
                                    int32_t* offsets, int32_t* row_token, int32_t* row_slot,
                                    int32_t* slot_row, int32_t* plan, uint32_t* err, cudaStream_t s) {
  return launch_pdl(permute_small_kernel, dim3(1), dim3(1024), 0, s, logits, w, idx, T, E, k, offsets,
                    row_token, row_slot, slot_row, plan, err);
}

cudaError_t launch_plan(const int32_t* offsets, int E, int rows_max, int32_t* plan, uint32_t* err,
                        cudaStream_t s) {
  plan_kernel<<<1, 1024, 0, s>>>(offsets, E, rows_max, plan, err);
  return cudaGetLastError();
}

}  // namespace k3moe
