// Routing: top-k selection with renormalised weights, the token-by-expert permutation, and
// the schedule ("plan") the expert kernels read.
//
// "kimi-k3-mlx", Architecture table: each token activates 16 of 896 routed experts.
// Selection keeps the k largest logits; equal logits go to the lower expert index (NaN
// ranks below every number, -0 equals +0). The kept indices are written in ascending order
// and their weights are the softmax over the kept logits, which equals softmax over all
// logits renormalised over the kept ones.
//
// Top-k: one CTA per token, a radix select over order-preserving 32-bit keys of the logits.
// Permutation: rows grouped by expert, token order inside an expert (the order a stable
// counting sort gives). Histogram -> exclusive scan -> scatter; the scatter walks tokens in
// chunks of 32 (one per lane) and ranks a (token, expert) pair inside its chunk with a
// per-expert lane bitmask, so the result is exact and deterministic.
#include "k3moe_device.cuh"
#include "k3moe_internal.cuh"
#include "k3moe_select.cuh"

namespace k3moe {
namespace {

__global__ void __launch_bounds__(kTopkThreads) topk_block_kernel(const float* __restrict__ logits, int T, int E,
                                                                  int k, int32_t* idx, float* w) {
  pdl_wait();
  pdl_trigger();
  if (blockIdx.x >= T) return;  // block-uniform
  block_topk(logits, blockIdx.x, E, k, idx, w);
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
// chunks of up to big_rows rows for the tensor-core expert GEMM. rows_max = T * k fixes
// where the second table sits. The second table lists the chunks of the experts with more than
// kSmallExpertRows rows first, then the other experts' chunks of up to kGemvTokens rows; its
// header is {chunks, chunks of the first kind, 0, 0}.
__device__ void build_plan(const int* off, int E, int rows_max, int32_t* plan, int* tmp, int* flag,
                           int* chunks, int big_rows) {
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
  const bool big = m > kSmallExpertRows;
  if (tid < E) {
    flag[tid] = big ? (m + big_rows - 1) / big_rows : 0;
    chunks[tid] = (m > 0 && !big) ? (m + kGemvTokens - 1) / kGemvTokens : 0;
  }
  __syncthreads();
  const int Cbig = block_excl_scan(flag, E, tmp);
  const int Csmall = block_excl_scan(chunks, E, tmp);
  if (tid < E && big)
    for (int q = 0; q * big_rows < m; ++q)
      ctab64[1 + flag[tid] + q] = make_int4(tid, off[tid] + q * big_rows, min(big_rows, m - q * big_rows), 0);
  if (tid < E && !big)
    for (int q = 0; q * kGemvTokens < m; ++q)
      ctab64[1 + Cbig + chunks[tid] + q] =
          make_int4(tid, off[tid] + q * kGemvTokens, min(kGemvTokens, m - q * kGemvTokens), 0);
  if (tid == 0) ctab64[0] = make_int4(Cbig + Csmall, Cbig, 0, 0);
}

// Scatter of tokens [t0, t1) by one warp, given base[e] = first free row of each expert.
__device__ void warp_scatter(const int32_t* __restrict__ idx, int t0, int t1, int E, int k,
                             int* base, unsigned* mask, int32_t* row_token, int32_t* row_slot,
                             int32_t* slot_row, uint32_t* err) {
  constexpr int kHalfK = 16;  // a token's slots are handled 16 at a time (k <= 32)
  const int lane = threadIdx.x & 31;
  const unsigned lt = (1u << lane) - 1u;
  for (int c0 = t0; c0 < t1; c0 += 32) {
    const int t = c0 + lane;
    const bool v = t < t1;
    // slots j0..j0+15 of this lane's token, read in one go (-1: none or out of range)
    auto load = [&](int j0, int (&ev)[kHalfK], bool report) {
#pragma unroll
      for (int q = 0; q < kHalfK; ++q) {
        const int j = j0 + q;
        const int e = (v && j < k) ? idx[(size_t)t * k + j] : -1;
        if (report && v && j < k && (e < 0 || e >= E)) atomicOr(err, kErrIndex);
        ev[q] = (e >= 0 && e < E) ? e : -1;
      }
    };
    int ev[kHalfK];
    for (int j0 = 0; j0 < k; j0 += kHalfK) {
      load(j0, ev, true);
#pragma unroll
      for (int q = 0; q < kHalfK; ++q)
        if (ev[q] >= 0) atomicOr(&mask[ev[q]], 1u << lane);
    }
    __syncwarp();
    for (int j0 = 0; j0 < k; j0 += kHalfK) {
      load(j0, ev, false);
#pragma unroll
      for (int q = 0; q < kHalfK; ++q) {
        if (ev[q] >= 0) {
          const int r = base[ev[q]] + __popc(mask[ev[q]] & lt);
          row_token[r] = t;
          row_slot[r] = j0 + q;
          slot_row[(size_t)t * k + j0 + q] = r;
        }
      }
    }
    __syncwarp();
    for (int j0 = 0; j0 < k; j0 += kHalfK) {
      load(j0, ev, false);
#pragma unroll
      for (int q = 0; q < kHalfK; ++q) {
        if (ev[q] >= 0) {
          const unsigned m = mask[ev[q]];
          if ((m & lt) == 0u) {  // lowest lane holding e advances its base and clears
            base[ev[q]] += __popc(m);
            mask[ev[q]] = 0u;
          }
        }
      }
    }
    __syncwarp();
  }
}

// ---------------------------------------------------------------- single-CTA permutation
// For T * k small: histogram, scan, scatter and plan in one block of 1024 threads (the indices
// pass through shared memory when T * k <= kSmallIdx).
constexpr int kSmallIdx = 2048;
__global__ void __launch_bounds__(1024) permute_small_kernel(const int32_t* idx, int T, int E, int k,
                                                             int32_t* offsets, int32_t* row_token,
                                                             int32_t* row_slot, int32_t* slot_row,
                                                             int32_t* plan, int* zcnt, int nzcnt, uint32_t* err,
                                                             int big_rows) {
  __shared__ int cnt[kMaxE + 1];
  __shared__ int tmp[1024];
  __shared__ int flag[kMaxE];
  __shared__ int chunks[kMaxE];
  __shared__ unsigned mask[kMaxE];
  __shared__ int s_idx[kSmallIdx];
  const int tid = threadIdx.x;
  pdl_wait();
  pdl_trigger();
  for (int i = tid; i < nzcnt; i += blockDim.x) zcnt[i] = 0;  // the decode expert kernel's counters
  const bool in_smem = T * k <= kSmallIdx;
  if (in_smem)
    for (int i = tid; i < T * k; i += blockDim.x) s_idx[i] = idx[i];
  if (tid <= E) cnt[tid] = 0;
  if (tid < E) mask[tid] = 0u;
  __syncthreads();
  const int32_t* ix = in_smem ? s_idx : idx;
  for (int i = tid; i < T * k; i += blockDim.x) {
    const int e = ix[i];
    if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);
  }
  __syncthreads();
  const int total = block_excl_scan(cnt, E, tmp);
  if (tid == 0) cnt[E] = total;
  __syncthreads();
  if (tid <= E) offsets[tid] = cnt[tid];
  __syncthreads();
  // plan reads the offsets before the scatter turns cnt into running bases
  build_plan(cnt, E, T * k, plan, tmp, flag, chunks, big_rows);
  __syncthreads();
  if (tid < 32) warp_scatter(ix, 0, T, E, k, cnt, mask, row_token, row_slot, slot_row, err);
}

// ---------------------------------------------------------------- a few tokens: top-k + permutation
// For T * k <= kTinyRows: each block selects one token's experts; the block that finishes last
// (a counter in the workspace, release/acquire through fences) builds the permutation and the
// plan, so decode pays for one kernel here instead of two.
constexpr int kTinyRows = 64;

// rows r = t * k + j (r < R <= kTinyRows), experts idx[r]: sorted rows grouped by expert, token
// order inside an expert; the same outputs as the histogram / scan / scatter path. All threads
// of the block take part.
// own_e >= 0: thread tid's expert is own_e (one token: this block selected it), not re-read from idx.
__device__ void block_route_tiny(const int32_t* idx, int T, int E, int k, int rows_max, int32_t* offsets,
                                 int32_t* row_token, int32_t* row_slot, int32_t* slot_row, int32_t* plan,
                                 uint32_t* err, int own_e = -1) {
  __shared__ uint32_t s_key[kTinyRows];
  __shared__ int s_e[kTinyRows], s_start[kTinyRows], s_run[kTinyRows + 1], s_chunks[kTinyRows];
  const int tid = threadIdx.x;
  const int R = T * k;
  // key = expert * kTinyRows + row: in key order, rows go by expert, then by row (token order)
  bool valid = false;
  if (tid < R) {
    const int e = own_e >= 0 ? own_e : __ldcg(idx + tid);
    valid = e >= 0 && e < E;
    if (!valid) {
      atomicOr(err, kErrIndex);
      slot_row[tid] = -1;  // contributes nothing to the combine
    }
    s_key[tid] = valid ? (uint32_t)e * kTinyRows + (uint32_t)tid : 0xffffffffu;
  }
  const int nvalid = __syncthreads_count(valid);
  if (valid) {
    const uint32_t key = s_key[tid];
    int p = 0;  // rank among the keys (distinct)
    for (int x = 0; x < R; ++x) p += s_key[x] < key ? 1 : 0;
    const int t = tid / k;
    row_token[p] = t;
    row_slot[p] = tid - t * k;
    slot_row[tid] = p;
    s_e[p] = (int)(key / kTinyRows);
  }
  __syncthreads();
  if (tid < nvalid) s_start[tid] = (tid == 0 || s_e[tid] != s_e[tid - 1]) ? 1 : 0;
  // offsets[e] = rows of experts below e
  for (int e = tid; e <= E; e += blockDim.x) {
    int lo = 0, hi = nvalid;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (s_e[mid] < e) lo = mid + 1; else hi = mid;
    }
    offsets[e] = lo;
  }
  __syncthreads();
  // runs of one expert = the active experts, in expert order
  int D = 0;
  for (int x = 0; x < nvalid; ++x) D += s_start[x];
  if (tid < nvalid && s_start[tid]) {
    int i = 0;
    for (int x = 0; x < tid; ++x) i += s_start[x];
    s_run[i] = tid;
  }
  if (tid == 0) s_run[D] = nvalid;
  __syncthreads();
  if (tid < D) s_chunks[tid] = (s_run[tid + 1] - s_run[tid] + kGemvTokens - 1) / kGemvTokens;
  __syncthreads();
  if (tid < D) {
    int C0 = 0;
    for (int x = 0; x < tid; ++x) C0 += s_chunks[x];
    const int p0 = s_run[tid], m = s_run[tid + 1] - p0, e = s_e[p0];
    int4* ctab = plan_ctab(plan, E);
    plan[2 + tid] = e;
    plan[2 + E + tid] = C0;
    for (int q = 0; q * kGemvTokens < m; ++q)
      ctab[C0 + q] = make_int4(e, p0 + q * kGemvTokens, min(kGemvTokens, m - q * kGemvTokens), 0);
    plan_ctab64(plan, E, rows_max)[1 + tid] = make_int4(e, p0, m, 0);  // m <= kTinyRows: one chunk
    if (tid == D - 1) {
      plan[0] = D;
      plan[1] = C0 + s_chunks[tid];
      plan[2 + E + D] = C0 + s_chunks[tid];
      plan_ctab64(plan, E, rows_max)[0] = make_int4(D, 0, 0, 0);
    }
  }
  if (D == 0 && tid == 0) {
    plan[0] = 0;
    plan[1] = 0;
    plan[2 + E] = 0;
    plan_ctab64(plan, E, rows_max)[0] = make_int4(0, 0, 0, 0);
  }
}

__global__ void __launch_bounds__(kTopkThreads) route_tiny_kernel(const float* __restrict__ logits, int T, int E,
                                                                  int k, int32_t* idx, float* w, int32_t* offsets,
                                                                  int32_t* row_token, int32_t* row_slot,
                                                                  int32_t* slot_row, int32_t* plan, int* done,
                                                                  int* cnt, int ncnt, uint32_t* err) {
  __shared__ int s_last;
  pdl_wait();
  pdl_trigger();
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < ncnt; i += blockDim.x) cnt[i] = 0;
  const int own_e = block_topk(logits, blockIdx.x, E, k, idx, w);
  if (T == 1) {  // the only block is the last: no count, and its own selection stays in registers
    if (__syncthreads_or(threadIdx.x < k && (own_e < 0 || own_e >= E)))
      block_route_tiny(idx, T, E, k, k, offsets, row_token, row_slot, slot_row, plan, err, own_e);
    else
      route_one_token(E, k, own_e, offsets, row_token, row_slot, slot_row, plan);
    return;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();  // this token's indices are visible before it is counted
    const int last = atomicAdd(done, 1) == T - 1;
    if (last) {
      *done = 0;  // ready for the next launch
      __threadfence();
    }
    s_last = last;
  }
  __syncthreads();
  if (s_last) block_route_tiny(idx, T, E, k, T * k, offsets, row_token, row_slot, slot_row, plan, err);
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
                                                    int32_t* offsets, int32_t* plan, int big_rows) {
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
  build_plan(cnt, E, rows_max, plan, tmp, flag, chunks, big_rows);
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
                                                    int rows_max, int32_t* plan, uint32_t* err, int big_rows) {
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
  build_plan(off, E, rows_max, plan, tmp, flag, chunks, big_rows);
}

}  // namespace

cudaError_t launch_topk(const float* logits, int T, int E, int k, int32_t* idx, float* w,
                        cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  return launch_pdl(topk_block_kernel, dim3(T), dim3(kTopkThreads), 0, s, logits, T, E, k, idx, w);
}

cudaError_t launch_permute(const int32_t* idx, int T, int E, int k, int32_t* offsets,
                           int32_t* row_token, int32_t* row_slot, int32_t* slot_row,
                           int32_t* plan, int32_t* scratch, uint32_t* err, cudaStream_t s, int big_rows) {
  if (T <= kBlockTokens) {
    permute_small_kernel<<<1, 1024, 0, s>>>(idx, T, E, k, offsets, row_token, row_slot, slot_row, plan, nullptr,
                                            0, err, big_rows);
    return cudaGetLastError();
  }
  const int nblk = (T + kBlockTokens - 1) / kBlockTokens;
  hist_kernel<<<nblk, 256, 0, s>>>(idx, T, E, k, scratch);
  scan_kernel<<<1, 1024, 0, s>>>(scratch, nblk, E, T * k, offsets, plan, big_rows);
  scatter_kernel<<<nblk, 32, 0, s>>>(idx, T, E, k, scratch, row_token, row_slot, slot_row, err);
  return cudaGetLastError();
}

cudaError_t launch_route_tail_small(const float* logits, int T, int E, int k, int32_t* idx, float* w,
                                    int32_t* offsets, int32_t* row_token, int32_t* row_slot,
                                    int32_t* slot_row, int32_t* plan, int* done, int* cnt, int ncnt,
                                    uint32_t* err, cudaStream_t s) {
  if (T * k <= kTinyRows)
    return launch_pdl(route_tiny_kernel, dim3(T), dim3(kTopkThreads), 0, s, logits, T, E, k, idx, w, offsets,
                      row_token, row_slot, slot_row, plan, done, cnt, ncnt, err);
  cudaError_t e = launch_pdl(topk_block_kernel, dim3(T), dim3(kTopkThreads), 0, s, logits, T, E, k, idx, w);
  if (e != cudaSuccess) return e;
  return launch_pdl(permute_small_kernel, dim3(1), dim3(1024), 0, s, (const int32_t*)idx, T, E, k, offsets,
                    row_token, row_slot, slot_row, plan, cnt, ncnt, err, (int)kUmmaChunkRows);
}

cudaError_t launch_plan(const int32_t* offsets, int E, int rows_max, int32_t* plan, uint32_t* err,
                        cudaStream_t s, int big_rows) {
  plan_kernel<<<1, 1024, 0, s>>>(offsets, E, rows_max, plan, err, big_rows);
  return cudaGetLastError();
}

}  // namespace k3moe
