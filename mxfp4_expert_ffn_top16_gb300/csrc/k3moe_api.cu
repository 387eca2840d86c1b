// C entry points of libk3moe (declared in include/k3moe.h): argument checks, workspace
// layout and the launch sequence of each call. Every device step runs in this library's
// kernels; nothing here computes on the host.
#include <cstdint>
#include <cstring>
#include <atomic>
#include <mutex>
#include <new>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "k3moe.h"
#include "k3moe_device.cuh"
#include "k3moe_internal.cuh"

namespace k3moe {

int num_sms() {
  static std::atomic<int> cached[64];  // zero-initialised (static storage); 0 = not yet queried
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

cudaError_t ensure_smem_attr(const void* fn, size_t bytes) {
  struct Rec { const void* fn; int dev; size_t bytes; };
  static Rec recs[64];
  static int n = 0;
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n; ++i)
    if (recs[i].fn == fn && recs[i].dev == dev && recs[i].bytes >= bytes) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  for (int i = 0; i < n; ++i)
    if (recs[i].fn == fn && recs[i].dev == dev) {
      recs[i].bytes = bytes;
      return e;
    }
  if (n < 64) recs[n++] = Rec{fn, dev, bytes};
  return e;
}

static size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

WsLayout ws_layout(const k3moe_dims& d, int64_t T) {
  WsLayout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += align256(bytes);
    return o;
  };
  const size_t E = (size_t)d.n_experts, k = (size_t)d.top_k, Lw = (size_t)d.latent,
               I = (size_t)d.inter, Tt = (size_t)T;
  const size_t rows = Tt * k;
  L.err = take(256);
  L.logits = take(Tt * E * 4);
  L.idx = take(rows * 4);
  L.wts = take(rows * 4);
  L.offsets = take((E + 1) * 4);
  L.row_token = take(rows * 4);
  L.row_slot = take(rows * 4);
  L.slot_row = take(rows * 4);
  L.plan = take(plan_bytes((int)E, (long long)rows));
  L.z = take(Tt * Lw * 2);
  L.zh = take(Tt * Lw * 2);
  L.zs = take(Tt * (size_t)exp_pitch(d.latent));
  L.a = take(rows * I * 2);
  L.ah = take(rows * I * 2);
  L.as = take(rows * (size_t)exp_pitch(d.inter));
  L.o = take(rows * Lw * 4);
  L.c = take(Tt * Lw * 2);
  L.xin = take(Tt * (size_t)d.hidden * 2);
  L.yout = take(Tt * (size_t)d.hidden * 2);
  L.perm = take(((Tt + 255) / 256) * E * 4);
  // the routing kernel's count of finished blocks must read zero at every launch, whatever T
  // the previous call on this workspace had: it sits in the fixed header, after the error word
  L.route_done = L.err + 4;
  {  // shared experts: gate and up (fp32), GLU output (bf16) [T][S]
    const size_t S = (size_t)d.n_shared * (size_t)d.shared_inter;
    L.sg = take(Tt * S * 4);
    L.su = take(Tt * S * 4);
    L.sa = take(Tt * S * 2);
  }
  if (umma_expert_ok(d)) {
    // P activation rows per sorted row (bf16 as e4m3 hi + lo: 2; MXFP8: 1) of one byte per value,
    // or for MXFP4 activations one row of packed e2m1 codes (half a byte per value)
    const size_t P = d.actq ? 1 : 2, num = d.actq == 2 ? 1 : 2;
    L.bq = take(P * rows * Lw * num / 2);
    L.bs = take(P * rows * (size_t)exp_pitch(d.latent));
    L.aq = take(P * rows * I * num / 2);
    L.aqs = take(P * rows * (size_t)exp_pitch(d.inter));
    L.chunk_done = take((size_t)decode_counters(d, T) * 4);
  }
  L.total = off;
  return L;
}

}  // namespace k3moe

using namespace k3moe;

namespace {

template <typename P>
P* at(void* ws, size_t off) {
  return reinterpret_cast<P*>(static_cast<uint8_t*>(ws) + off);
}

bool misaligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

k3moe_status check_dims(const k3moe_dims* d) {
  if (!d) return K3MOE_E_NULL;
  if (d->hidden <= 0 || d->latent <= 0 || d->inter <= 0) return K3MOE_E_SHAPE;
  if (d->hidden % 64 || d->latent % 64 || d->inter % 64) return K3MOE_E_SHAPE;
  if (d->n_experts < 1 || d->n_experts > 1024) return K3MOE_E_SHAPE;
  if (d->top_k < 1 || d->top_k > 32 || d->top_k > d->n_experts) return K3MOE_E_SHAPE;
  if (d->act != 0) return K3MOE_E_MODE;
  if (d->actq < 0 || d->actq > 2) return K3MOE_E_MODE;
  // MXFP4 activations run on the kind::mxf4 tensor-core path only: K = 256 per stage
  if (d->actq == 2 && (d->latent % 256 || d->inter % 256)) return K3MOE_E_MODE;
  if (d->n_shared < 0 || d->n_shared > 8) return K3MOE_E_SHAPE;
  if (d->n_shared > 0 && (d->shared_inter <= 0 || ((int64_t)d->n_shared * d->shared_inter) % 64 ||
                          (int64_t)d->n_shared * d->shared_inter > (1 << 20)))
    return K3MOE_E_SHAPE;
  return K3MOE_OK;
}

k3moe_status check_ws(const k3moe_dims& d, int32_t T, void* ws, size_t ws_bytes) {
  if (!ws) return K3MOE_E_WORKSPACE;
  if (misaligned(ws)) return K3MOE_E_ALIGN;
  if (ws_layout(d, T).total > ws_bytes) return K3MOE_E_WORKSPACE;
  return K3MOE_OK;
}

k3moe_status check_weights(const k3moe_weights* w, bool dense, bool experts) {
  if (!w) return K3MOE_E_NULL;
  if (dense) {
    if (!w->w_router || !w->w_in || !w->w_out) return K3MOE_E_NULL;
    if (misaligned(w->w_router) || misaligned(w->w_in) || misaligned(w->w_out) ||
        misaligned(w->router_bias))
      return K3MOE_E_ALIGN;
  }
  if (experts) {
    const void* p[6] = {w->gate_q, w->gate_s, w->up_q, w->up_s, w->down_q, w->down_s};
    for (const void* q : p) {
      if (!q) return K3MOE_E_NULL;
      if (misaligned(q)) return K3MOE_E_ALIGN;
    }
  }
  return K3MOE_OK;
}

k3moe_status check_shared(const k3moe_dims& d, const k3moe_weights* w) {
  if (d.n_shared == 0) return K3MOE_OK;
  const void* p[3] = {w->w_shared_gate, w->w_shared_up, w->w_shared_down};
  for (const void* q : p) {
    if (!q) return K3MOE_E_NULL;
    if (misaligned(q)) return K3MOE_E_ALIGN;
  }
  return K3MOE_OK;
}

// ---------------------------------------------------------------- diagnostic profiling
enum ProfId {
  P_ROUTER_LATENT = 0, P_TOPK, P_PERMUTE, P_GLU, P_DOWN, P_COMBINE, P_LATENT_OUT, P_QUANT,
  P_GLU_MMA, P_DOWN_MMA, P_FFN_MMA, P_SHARED, P_COUNT
};
const char* const kProfNames[P_COUNT] = {"router_latent_in", "topk", "permute",
                                         "expert_glu_gemv", "expert_down_gemv", "combine",
                                         "latent_out", "expert_act_quant", "expert_glu_mma",
                                         "expert_down_mma", "expert_ffn_mma", "shared_experts"};
struct Profiler {
  bool on = false;
  static constexpr int kMax = 65536;
  cudaEvent_t* ev = nullptr;  // pairs
  int* id = nullptr;
  int used = 0;
};
Profiler g_prof;

struct ProfScope {
  int slot = -1;
  cudaStream_t s;
  ProfScope(int pid, cudaStream_t st) : s(st) {
    if (!g_prof.on || g_prof.used >= Profiler::kMax) return;
    slot = g_prof.used++;
    g_prof.id[slot] = pid;
    cudaEventRecord(g_prof.ev[2 * slot], s);
  }
  ~ProfScope() {
    if (slot >= 0) cudaEventRecord(g_prof.ev[2 * slot + 1], s);
  }
};

#define K3_TRY(expr)                        \
  do {                                      \
    const k3moe_status st_ = (expr);        \
    if (st_ != K3MOE_OK) return st_;        \
  } while (0)
#define K3_CUDA(expr)                                  \
  do {                                                 \
    if ((expr) != cudaSuccess) return K3MOE_E_CUDA;    \
  } while (0)

// Expert GEMMs for the sorted rows (plan already built): block-scaled tensor-core tiles for
// many tokens, the GEMV on f16 copies (zh, zs already in ws) otherwise.
// z_rows_ready: (decode, tensor-core path) the dense kernel already wrote z as P E4M3 rows per
// token into bq / bs, and the routing kernel cleared the chunk counters.
k3moe_status run_expert_gemms(const k3moe_dims& d, const k3moe_weights& w, const uint16_t* z, int32_t T,
                              const int32_t* offsets, const int32_t* row_token, float* o_rows, void* ws,
                              const WsLayout& L, cudaStream_t s, bool z_rows_ready = false,
                              const PackedScales* ps = nullptr, const DecodeSelect* sel = nullptr,
                              const int32_t* slot_row = nullptr) {
  uint32_t* err = at<uint32_t>(ws, L.err);
  int32_t* plan = at<int32_t>(ws, L.plan);
  if (umma_expert_ok(d)) {
    // activation rows per sorted row: 2 (bf16 as e4m3 hi + lo), 1 (MXFP8), 0 = one MXFP4 row
    const int P = d.actq == 2 ? 0 : (d.actq ? 1 : 2);
    int* cnt = at<int>(ws, L.chunk_done);
    uint8_t* aq = at<uint8_t>(ws, L.aq);
    uint8_t* aqs = at<uint8_t>(ws, L.aqs);
    if (T < kUmmaExpertMinTokens && P != 0) {
      // decode: z as P E4M3 rows per token (the expert kernel gathers a chunk's rows by token);
      // both passes in one launch (on the N side when latent % 256 == 0)
      if (!z_rows_ready) {
        ProfScope p(P_QUANT, s);
        K3_CUDA(launch_quant_rows(z, nullptr, T, T, d.latent, P, at<uint8_t>(ws, L.bq), at<uint8_t>(ws, L.bs),
                                  cnt, decode_counters(d, T), err, s));
      }
      if (decode_weights_on_m(P, T)) {
        ProfScope p(P_FFN_MMA, s);
        K3_CUDA(launch_umma_decode(d, w, ps, plan, at<uint8_t>(ws, L.bq), at<uint8_t>(ws, L.bs), row_token, P, T,
                                   aq, aqs, o_rows, cnt, err, s, sel));
      } else {
        const bool both = d.latent % 256 == 0;
        {
          ProfScope p(both ? P_FFN_MMA : P_GLU_MMA, s);
          K3_CUDA(launch_umma_wn(d, w, ps, plan, at<uint8_t>(ws, L.bq), at<uint8_t>(ws, L.bs), row_token, P, T, aq,
                                 aqs, both, o_rows, cnt, err, s));
        }
        if (!both) {
          ProfScope p(P_DOWN_MMA, s);
          K3_CUDA(launch_umma_down(d, w, plan, aq, aqs, P, T, o_rows, err, s));
        }
      }
      return K3MOE_OK;
    }
    // Many tokens with e4m3 activations: the experts with at most kSmallExpertRows rows (one
    // chunk each) run on the weights-on-N decode kernel, which streams a weight tile for a few
    // rows at a far higher rate than the many-token tiles; the others on the many-token kernel.
    const bool small_split = T >= kUmmaExpertMinTokens && P != 0 && d.latent % 256 == 0;
    {  // many tokens (and MXFP4 activations at any count): z gathered into rows per sorted row
      ProfScope p(P_QUANT, s);
      // (with the permutation's slot -> row table: each token converted once, stored to its k rows)
      K3_CUDA(launch_quant_rows(z, row_token, T * d.top_k, T, d.latent, P, at<uint8_t>(ws, L.bq),
                                at<uint8_t>(ws, L.bs), cnt, small_split ? decode_counters(d, T) : 0, err, s,
                                slot_row, d.top_k));
    }
    {
      ProfScope p(P_GLU_MMA, s);
      K3_CUDA(launch_umma_glu(d, w, plan, at<uint8_t>(ws, L.bq), at<uint8_t>(ws, L.bs), P, T, aq, aqs, err, s,
                              small_split, ps));
    }
    {
      ProfScope p(P_DOWN_MMA, s);
      K3_CUDA(launch_umma_down(d, w, plan, aq, aqs, P, T, o_rows, err, s, small_split, ps));
    }
    if (small_split) {
      ProfScope p(P_FFN_MMA, s);
      K3_CUDA(launch_umma_wn(d, w, ps, plan, at<uint8_t>(ws, L.bq), at<uint8_t>(ws, L.bs), nullptr, P, T, aq, aqs,
                             true, o_rows, cnt, err, s, true));
    }
    return K3MOE_OK;
  }
  {
    ProfScope p(P_GLU, s);
    K3_CUDA(launch_expert_glu(d, w, plan, offsets, row_token, at<__half>(ws, L.zh), at<int8_t>(ws, L.zs),
                              at<uint16_t>(ws, L.a), at<__half>(ws, L.ah), at<int8_t>(ws, L.as), T, err, s));
  }
  ProfScope p(P_DOWN, s);
  K3_CUDA(launch_expert_down(d, w, plan, offsets, at<__half>(ws, L.ah), at<int8_t>(ws, L.as), o_rows, T, err,
                             s));
  return K3MOE_OK;
}

// Route + permute + experts + combine for T tokens whose logits / z are already in ws.
// One token on the tensor-core expert kernel with the weights on M: that kernel selects the
// experts itself (the dense kernel before it clears its counters), no routing kernel runs.
inline bool decode_select_in_experts(const k3moe_dims& d, int32_t T) {
  return T == 1 && umma_expert_ok(d) && d.actq != 2 && decode_weights_on_m(d.actq ? 1 : 2, T) &&
         T < kUmmaDenseMinTokens && d.top_k <= 32;
}

// Bytes of the latent-out weight the one-token expert kernel fetches into L2 ahead of its use.
inline long long l2_next_bytes(const k3moe_dims& d) {
  const long long b = (long long)d.hidden * d.latent * 2;
  return (long long)(kL2NextFraction * (double)b) / 256 * 256;
}

k3moe_status run_experts_decode(const k3moe_dims& d, const k3moe_weights& w, int32_t T, void* ws,
                                const WsLayout& L, int32_t* idx, float* wts, cudaStream_t s,
                                const PackedScales* ps) {
  uint32_t* err = at<uint32_t>(ws, L.err);
  const bool fused_select = decode_select_in_experts(d, T);
  if (fused_select) {
    // (no routing kernel: the expert kernel selects the experts and writes the routing outputs)
  } else if (T <= kSmallRouteTokens) {
    ProfScope p(P_PERMUTE, s);  // top-k, then permutation and plan (one kernel for a few tokens)
    K3_CUDA(launch_route_tail_small(at<float>(ws, L.logits), T, d.n_experts, d.top_k, idx, wts,
                                    at<int32_t>(ws, L.offsets), at<int32_t>(ws, L.row_token),
                                    at<int32_t>(ws, L.row_slot), at<int32_t>(ws, L.slot_row),
                                    at<int32_t>(ws, L.plan), at<int>(ws, L.route_done),
                                    umma_expert_ok(d) ? at<int>(ws, L.chunk_done) : nullptr,
                                    umma_expert_ok(d) ? decode_counters(d, T) : 0, err, s));
  } else {
    {
      ProfScope p(P_TOPK, s);
      K3_CUDA(launch_topk(at<float>(ws, L.logits), T, d.n_experts, d.top_k, idx, wts, s));
    }
    ProfScope p(P_PERMUTE, s);
    K3_CUDA(launch_permute(idx, T, d.n_experts, d.top_k, at<int32_t>(ws, L.offsets),
                           at<int32_t>(ws, L.row_token), at<int32_t>(ws, L.row_slot),
                           at<int32_t>(ws, L.slot_row), at<int32_t>(ws, L.plan),
                           at<int32_t>(ws, L.perm), err, s, many_chunk_rows(d.actq)));
  }
  // (decode, tensor-core experts: the dense kernel wrote z's E4M3 rows, the routing cleared the
  // chunk counters)
  const DecodeSelect sel{at<float>(ws, L.logits), idx, wts, at<int32_t>(ws, L.offsets),
                         at<int32_t>(ws, L.row_token), at<int32_t>(ws, L.row_slot), at<int32_t>(ws, L.slot_row),
                         w.w_out, l2_next_bytes(d)};
  K3_TRY(run_expert_gemms(d, w, at<uint16_t>(ws, L.z), T, at<int32_t>(ws, L.offsets),
                          at<int32_t>(ws, L.row_token), at<float>(ws, L.o), ws, L, s,
                          T <= kSmallRouteTokens && T < kUmmaExpertMinTokens && T < kUmmaDenseMinTokens &&
                              umma_expert_ok(d) && d.actq != 2,
                          ps, fused_select ? &sel : nullptr, at<int32_t>(ws, L.slot_row)));
  {
    ProfScope p(P_COMBINE, s);
    K3_CUDA(launch_combine(at<float>(ws, L.o), at<int32_t>(ws, L.slot_row), wts, T, d.top_k,
                           d.latent, at<uint16_t>(ws, L.c), s));
  }
  return K3MOE_OK;
}

}  // namespace

extern "C" {

const char* k3moe_status_string(k3moe_status s) {
  switch (s) {
    case K3MOE_OK: return "K3MOE_OK";
    case K3MOE_E_NULL: return "K3MOE_E_NULL: a required pointer is NULL";
    case K3MOE_E_SHAPE: return "K3MOE_E_SHAPE: unsupported size";
    case K3MOE_E_ALIGN: return "K3MOE_E_ALIGN: pointer not 16-byte aligned";
    case K3MOE_E_WORKSPACE: return "K3MOE_E_WORKSPACE: workspace missing or too small";
    case K3MOE_E_MODE: return "K3MOE_E_MODE: unsupported activation or activation format";
    case K3MOE_E_CUDA: return "K3MOE_E_CUDA: CUDA call or launch failed";
    case K3MOE_E_TIMEOUT: return "K3MOE_E_TIMEOUT: a device-side bounded wait ran out";
    case K3MOE_E_DEVICE: return "K3MOE_E_DEVICE: device-side check failed";
    case K3MOE_E_SCRATCH:
      return "K3MOE_E_SCRATCH: T * n_experts exceeds the 65536 logits of k3moe_route_noalloc's fixed scratch";
    case K3MOE_E_HOSTMEM:
      return "K3MOE_E_HOSTMEM: a host buffer is not page-locked memory the device can address";
  }
  return "K3MOE: unknown status";
}

k3moe_status k3moe_workspace_size(const k3moe_dims* dims, int32_t max_tokens, size_t* bytes) {
  K3_TRY(check_dims(dims));
  if (!bytes) return K3MOE_E_NULL;
  if (max_tokens < 0) return K3MOE_E_SHAPE;
  *bytes = ws_layout(*dims, max_tokens).total;
  return K3MOE_OK;
}

k3moe_status k3moe_route(const k3moe_dims* dims, const uint16_t* x, int32_t T,
                         const uint16_t* w_router, const float* bias, float* logits,
                         int32_t* topk_idx, float* topk_w, void* ws, size_t ws_bytes,
                         void* stream) {
  K3_TRY(check_dims(dims));
  const k3moe_dims& d = *dims;
  if (T < 0) return K3MOE_E_SHAPE;
  if (!x || !w_router || !topk_idx || !topk_w) return K3MOE_E_NULL;
  if (misaligned(x) || misaligned(w_router) || misaligned(bias) || misaligned(logits) ||
      misaligned(topk_idx) || misaligned(topk_w))
    return K3MOE_E_ALIGN;
  K3_TRY(check_ws(d, T, ws, ws_bytes));
  if (T == 0) return K3MOE_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const WsLayout L = ws_layout(d, T);
  float* lg = logits ? logits : at<float>(ws, L.logits);
  K3_CUDA(launch_dense(w_router, d.n_experts, lg, nullptr, bias, nullptr, 0, nullptr, nullptr,
                            nullptr, 0, x, T, d.hidden, at<uint32_t>(ws, L.err), s));
  K3_CUDA(launch_topk(lg, T, d.n_experts, d.top_k, topk_idx, topk_w, s));
  return K3MOE_OK;
}

k3moe_status k3moe_permute(const k3moe_dims* dims, const int32_t* topk_idx, int32_t T,
                           int32_t* expert_offsets, int32_t* row_token, int32_t* row_slot,
                           int32_t* slot_row, void* ws, size_t ws_bytes, void* stream) {
  K3_TRY(check_dims(dims));
  const k3moe_dims& d = *dims;
  if (T < 0) return K3MOE_E_SHAPE;
  if (!topk_idx || !expert_offsets || !row_token || !row_slot || !slot_row) return K3MOE_E_NULL;
  if (misaligned(topk_idx) || misaligned(expert_offsets) || misaligned(row_token) ||
      misaligned(row_slot) || misaligned(slot_row))
    return K3MOE_E_ALIGN;
  K3_TRY(check_ws(d, T, ws, ws_bytes));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const WsLayout L = ws_layout(d, T);
  K3_CUDA(launch_permute(topk_idx, T, d.n_experts, d.top_k, expert_offsets, row_token, row_slot,
                         slot_row, at<int32_t>(ws, L.plan), at<int32_t>(ws, L.perm),
                         at<uint32_t>(ws, L.err), s, many_chunk_rows(d.actq)));
  return K3MOE_OK;
}

k3moe_status k3moe_project(const uint16_t* W, const uint16_t* x, int32_t T, int32_t N, int32_t K,
                           uint16_t* out, void* ws, size_t ws_bytes, void* stream) {
  if (!W || !x || !out) return K3MOE_E_NULL;
  if (T < 0 || N <= 0 || K <= 0 || N % 64 || K % 64) return K3MOE_E_SHAPE;
  if (misaligned(W) || misaligned(x) || misaligned(out)) return K3MOE_E_ALIGN;
  if (!ws || ws_bytes < 256) return K3MOE_E_WORKSPACE;
  if (misaligned(ws)) return K3MOE_E_ALIGN;
  if (T == 0) return K3MOE_OK;
  K3_CUDA(launch_dense(W, N, nullptr, out, nullptr, nullptr, 0, nullptr, nullptr, nullptr, 0,
                            x, T, K, static_cast<uint32_t*>(ws), static_cast<cudaStream_t>(stream)));
  return K3MOE_OK;
}

k3moe_status k3moe_expert_ffn_mxfp4(const k3moe_dims* dims, const k3moe_weights* weights,
                                    const uint16_t* z, int32_t T, const int32_t* expert_offsets,
                                    const int32_t* row_token, float* o_rows, void* ws,
                                    size_t ws_bytes, void* stream) {
  K3_TRY(check_dims(dims));
  const k3moe_dims& d = *dims;
  K3_TRY(check_weights(weights, false, true));
  if (T < 0) return K3MOE_E_SHAPE;
  if (!z || !expert_offsets || !row_token || !o_rows) return K3MOE_E_NULL;
  if (misaligned(z) || misaligned(expert_offsets) || misaligned(row_token) || misaligned(o_rows))
    return K3MOE_E_ALIGN;
  K3_TRY(check_ws(d, T, ws, ws_bytes));
  if (T == 0) return K3MOE_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const WsLayout L = ws_layout(d, T);
  uint32_t* err = at<uint32_t>(ws, L.err);
  if (!umma_expert_ok(d))
    K3_CUDA(launch_act_prep(z, T, d.latent, d.actq, at<__half>(ws, L.zh), at<int8_t>(ws, L.zs), s));
  K3_CUDA(launch_plan(expert_offsets, d.n_experts, T * d.top_k, at<int32_t>(ws, L.plan), err, s,
                      many_chunk_rows(d.actq)));
  K3_TRY(run_expert_gemms(d, *weights, z, T, expert_offsets, row_token, o_rows, ws, L, s));
  return K3MOE_OK;
}

k3moe_status k3moe_combine(const k3moe_dims* dims, const float* o_rows, const int32_t* slot_row,
                           const float* topk_w, int32_t T, uint16_t* c, void* stream) {
  K3_TRY(check_dims(dims));
  const k3moe_dims& d = *dims;
  if (T < 0) return K3MOE_E_SHAPE;
  if (!o_rows || !slot_row || !topk_w || !c) return K3MOE_E_NULL;
  if (misaligned(o_rows) || misaligned(slot_row) || misaligned(topk_w) || misaligned(c))
    return K3MOE_E_ALIGN;
  if (T == 0) return K3MOE_OK;
  K3_CUDA(launch_combine(o_rows, slot_row, topk_w, T, d.top_k, d.latent, c,
                         static_cast<cudaStream_t>(stream)));
  return K3MOE_OK;
}

}  // extern "C"

namespace {
k3moe_status layer_forward(const k3moe_dims* dims, const k3moe_weights* weights, const PackedScales* ps,
                           const uint16_t* x, int32_t T, uint16_t* y, int32_t* topk_idx_out, float* topk_w_out,
                           void* ws, size_t ws_bytes, void* stream) {
  K3_TRY(check_dims(dims));
  const k3moe_dims& d = *dims;
  K3_TRY(check_weights(weights, true, true));
  K3_TRY(check_shared(d, weights));
  if (T < 0) return K3MOE_E_SHAPE;
  if (!x || !y) return K3MOE_E_NULL;
  if (misaligned(x) || misaligned(y) || misaligned(topk_idx_out) || misaligned(topk_w_out))
    return K3MOE_E_ALIGN;
  K3_TRY(check_ws(d, T, ws, ws_bytes));
  if (T == 0) return K3MOE_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const WsLayout L = ws_layout(d, T);
  uint32_t* err = at<uint32_t>(ws, L.err);
  int32_t* idx = topk_idx_out ? topk_idx_out : at<int32_t>(ws, L.idx);
  float* wts = topk_w_out ? topk_w_out : at<float>(ws, L.wts);
  const k3moe_weights& w = *weights;
  // router logits and z = bf16(W_in x) in one pass over x (+ the f16 block-scaled copy of z
  // that the expert GEMV reads, or for decode on tensor cores z's E4M3 rows per token)
  {
    ProfScope p(P_ROUTER_LATENT, s);
    const bool f16_copy = !umma_expert_ok(d);
    // decode on the tensor-core experts: z also as P E4M3 rows per token for the expert kernel
    const bool rows = !f16_copy && d.actq != 2 && T <= kSmallRouteTokens && T < kUmmaExpertMinTokens &&
                      T < kUmmaDenseMinTokens;
    // (when the expert kernel selects the experts itself, this kernel clears its counters)
    const bool fused_select = decode_select_in_experts(d, T);
    K3_CUDA(launch_dense(w.w_router, d.n_experts, at<float>(ws, L.logits), nullptr, w.router_bias, w.w_in,
                         d.latent, at<uint16_t>(ws, L.z), f16_copy ? at<__half>(ws, L.zh) : nullptr,
                         f16_copy ? at<int8_t>(ws, L.zs) : nullptr, d.actq, x, T, d.hidden, err, s,
                         rows ? at<uint8_t>(ws, L.bq) : nullptr, rows ? at<uint8_t>(ws, L.bs) : nullptr,
                         d.actq ? 1 : 2, nullptr, nullptr, nullptr, 0,
                         fused_select ? at<int>(ws, L.chunk_done) : nullptr,
                         fused_select ? decode_counters(d, T) : 0));
  }
  K3_TRY(run_experts_decode(d, w, T, ws, L, idx, wts, s, ps));
  // shared experts on the residual: g, u = G x, U x (fp32); a = bf16(silu(g) u)
  const int S = d.n_shared * d.shared_inter;
  if (S > 0) {
    ProfScope p(P_SHARED, s);
    K3_CUDA(launch_dense(w.w_shared_gate, S, at<float>(ws, L.sg), nullptr, nullptr, w.w_shared_up, S, nullptr,
                         nullptr, nullptr, 0, x, T, d.hidden, err, s, nullptr, nullptr, 0, at<float>(ws, L.su)));
    K3_CUDA(launch_glu(at<float>(ws, L.sg), at<float>(ws, L.su), (long long)T * S, at<uint16_t>(ws, L.sa), s));
  }
  {  // y = bf16(W_out c + D a): the shared experts' down projection is a second K segment
    ProfScope p(P_LATENT_OUT, s);
    K3_CUDA(launch_dense(w.w_out, d.hidden, nullptr, y, nullptr, nullptr, 0, nullptr, nullptr,
                         nullptr, 0, at<uint16_t>(ws, L.c), T, d.latent, err, s, nullptr, nullptr, 0, nullptr,
                         S > 0 ? w.w_shared_down : nullptr, S > 0 ? at<uint16_t>(ws, L.sa) : nullptr, S));
  }
  return K3MOE_OK;
}
}  // namespace

// A prepared layer: the caller's dims and weight pointers, and the expert scales repacked for
// the decode expert kernel (device memory the handle owns).
struct k3moe_layer {
  k3moe_dims dims;
  k3moe_weights weights;
  void* packed;  // gate, up, down staging images back to back; null when the shapes have none
  PackedScales ps;
};

extern "C" {

k3moe_status k3moe_layer_forward(const k3moe_dims* dims, const k3moe_weights* weights,
                                 const uint16_t* x, int32_t T, uint16_t* y,
                                 int32_t* topk_idx_out, float* topk_w_out, void* ws,
                                 size_t ws_bytes, void* stream) {
  return layer_forward(dims, weights, nullptr, x, T, y, topk_idx_out, topk_w_out, ws, ws_bytes, stream);
}

k3moe_status k3moe_layer_init(const k3moe_dims* dims, const k3moe_weights* weights, k3moe_layer** layer,
                              void* stream) {
  if (!layer) return K3MOE_E_NULL;
  *layer = nullptr;
  K3_TRY(check_dims(dims));
  const k3moe_dims& d = *dims;
  K3_TRY(check_weights(weights, true, true));
  K3_TRY(check_shared(d, weights));
  k3moe_layer* h = new (std::nothrow) k3moe_layer();
  if (!h) return K3MOE_E_CUDA;
  h->dims = d;
  h->weights = *weights;
  if (umma_expert_ok(d)) {
    const size_t gbytes = (size_t)d.n_experts * d.inter * (d.latent / 32);
    const size_t dbytes = (size_t)d.n_experts * d.latent * (d.inter / 32);
    uint8_t* p = nullptr;
    if (cudaMalloc(&p, 4 * gbytes + dbytes) != cudaSuccess) {
      delete h;
      return K3MOE_E_CUDA;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const long long grows = (long long)d.n_experts * d.inter, drows = (long long)d.n_experts * d.latent;
    if (launch_pack_scales(weights->gate_s, grows, d.latent, p, s) != cudaSuccess ||
        launch_pack_scales(weights->up_s, grows, d.latent, p + gbytes, s) != cudaSuccess ||
        launch_pack_scales(weights->down_s, drows, d.inter, p + 2 * gbytes, s) != cudaSuccess ||
        launch_pack_scales_glu(weights->gate_s, weights->up_s, grows, d.latent, p + 2 * gbytes + dbytes, s) !=
            cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
      cudaFree(p);
      delete h;
      return K3MOE_E_CUDA;
    }
    h->packed = p;
    h->ps = PackedScales{p, p + gbytes, p + 2 * gbytes, p + 2 * gbytes + dbytes};
  }
  *layer = h;
  return K3MOE_OK;
}

k3moe_status k3moe_layer_free(k3moe_layer* layer) {
  if (!layer) return K3MOE_OK;
  const bool ok = !layer->packed || cudaFree(layer->packed) == cudaSuccess;
  delete layer;
  return ok ? K3MOE_OK : K3MOE_E_CUDA;
}

k3moe_status k3moe_layer_run(const k3moe_layer* layer, const uint16_t* x, int32_t T, uint16_t* y,
                             int32_t* topk_idx_out, float* topk_w_out, void* ws, size_t ws_bytes, void* stream) {
  if (!layer) return K3MOE_E_NULL;
  return layer_forward(&layer->dims, &layer->weights, layer->packed ? &layer->ps : nullptr, x, T, y, topk_idx_out,
                       topk_w_out, ws, ws_bytes, stream);
}

// The device address of page-locked host memory mapped into the device's address space; null
// for any other pointer (pageable, device or managed memory).
static void* host_device_ptr(const void* p) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

k3moe_status k3moe_layer_run_host(const k3moe_layer* layer, const uint16_t* x_host, int32_t T, uint16_t* y_host,
                                  int32_t* topk_idx_out, float* topk_w_out, void* ws, size_t ws_bytes,
                                  void* stream) {
  if (!layer) return K3MOE_E_NULL;
  const k3moe_dims& d = layer->dims;
  if (T < 0) return K3MOE_E_SHAPE;
  if (!x_host || !y_host) return K3MOE_E_NULL;
  K3_TRY(check_ws(d, T, ws, ws_bytes));
  if (T == 0) return K3MOE_OK;
  const size_t bytes = (size_t)T * d.hidden * 2;
  if (bytes % 16) return K3MOE_E_SHAPE;
  void* xd = host_device_ptr(x_host);
  void* yd = host_device_ptr(y_host);
  if (!xd || !yd) return K3MOE_E_HOSTMEM;
  if (misaligned(xd) || misaligned(yd)) return K3MOE_E_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const WsLayout L = ws_layout(d, T);
  uint16_t* xin = at<uint16_t>(ws, L.xin);
  uint16_t* yout = at<uint16_t>(ws, L.yout);
  K3_CUDA(launch_copy16(xd, xin, bytes, s));
  K3_TRY(layer_forward(&layer->dims, &layer->weights, layer->packed ? &layer->ps : nullptr, xin, T, yout,
                       topk_idx_out, topk_w_out, ws, ws_bytes, stream));
  K3_CUDA(launch_copy16(yout, yd, bytes, s));
  return K3MOE_OK;
}

k3moe_status k3moe_layer_saliency(const k3moe_dims* dims, int32_t T, const int32_t* topk_idx, const float* topk_w,
                                  void* ws, size_t ws_bytes, double* saliency, void* stream) {
  K3_TRY(check_dims(dims));
  const k3moe_dims& d = *dims;
  if (T < 0) return K3MOE_E_SHAPE;
  if (!saliency) return K3MOE_E_NULL;
  if (misaligned(topk_idx) || misaligned(topk_w) || misaligned(saliency)) return K3MOE_E_ALIGN;
  K3_TRY(check_ws(d, T, ws, ws_bytes));
  if (T == 0) return K3MOE_OK;
  const WsLayout L = ws_layout(d, T);
  K3_CUDA(launch_saliency(at<float>(ws, L.o), at<int32_t>(ws, L.row_token), at<int32_t>(ws, L.row_slot),
                          topk_idx ? topk_idx : at<int32_t>(ws, L.idx), topk_w ? topk_w : at<float>(ws, L.wts), T,
                          d.top_k, d.latent, d.n_experts, saliency, at<uint32_t>(ws, L.err),
                          static_cast<cudaStream_t>(stream)));
  return K3MOE_OK;
}

k3moe_status k3moe_profile(int32_t mode, int32_t n, float* total_ms, int32_t* launches) {
  if (mode == 1) {
    if (!g_prof.ev) {
      g_prof.ev = new cudaEvent_t[2 * Profiler::kMax];
      g_prof.id = new int[Profiler::kMax];
      for (int i = 0; i < 2 * Profiler::kMax; ++i)
        if (cudaEventCreate(&g_prof.ev[i]) != cudaSuccess) return K3MOE_E_CUDA;
    }
    g_prof.used = 0;
    g_prof.on = true;
    return K3MOE_OK;
  }
  g_prof.on = false;
  for (int i = 0; i < n; ++i) {
    if (total_ms) total_ms[i] = 0.f;
    if (launches) launches[i] = 0;
  }
  for (int j = 0; j < g_prof.used; ++j) {
    float ms = 0.f;
    if (cudaEventSynchronize(g_prof.ev[2 * j + 1]) != cudaSuccess) return K3MOE_E_CUDA;
    if (cudaEventElapsedTime(&ms, g_prof.ev[2 * j], g_prof.ev[2 * j + 1]) != cudaSuccess)
      return K3MOE_E_CUDA;
    const int i = g_prof.id[j];
    if (i < n) {
      if (total_ms) total_ms[i] += ms;
      if (launches) launches[i] += 1;
    }
  }
  g_prof.used = 0;
  return K3MOE_OK;
}

const char* k3moe_profile_name(int32_t id) {
  return (id >= 0 && id < P_COUNT) ? kProfNames[id] : nullptr;
}

k3moe_status k3moe_layer_stats(const k3moe_dims* dims, int32_t T, void* ws, size_t ws_bytes, void* stream,
                               int32_t* distinct, int64_t* expert_bytes) {
  K3_TRY(check_dims(dims));
  const k3moe_dims& d = *dims;
  if (T < 0) return K3MOE_E_SHAPE;
  K3_TRY(check_ws(d, T, ws, ws_bytes));
  int32_t D = 0;
  if (T > 0) {
    const WsLayout L = ws_layout(d, T);
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return K3MOE_E_CUDA;
    // plan[0]: active experts of the step, written by the routing / plan kernels
    if (cudaMemcpy(&D, at<int32_t>(ws, L.plan), sizeof(D), cudaMemcpyDeviceToHost) != cudaSuccess)
      return K3MOE_E_CUDA;
    if (D < 0 || D > d.n_experts) return K3MOE_E_DEVICE;
  }
  if (distinct) *distinct = D;
  if (expert_bytes) {  // per expert: gate and up codes + scales, down codes + scales
    const int64_t L_ = d.latent, I = d.inter;
    *expert_bytes = (int64_t)D * (2 * (I * L_ / 2 + I * L_ / 32) + (L_ * I / 2 + L_ * I / 32));
  }
  return K3MOE_OK;
}

}  // extern "C"

namespace k3moe {
namespace {
// One thread waits on a barrier nobody arrives on: mbar_wait_bounded gives up after its wall-clock
// limit, sets the timeout bit of *err and returns (the self test of the failure path).
__global__ void wait_selftest_kernel(uint32_t* err) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait_bounded(&bar, 0, &abort_flag, err);
}
}  // namespace
}  // namespace k3moe

extern "C" {

k3moe_status k3moe_selftest_timeout(void* ws, void* stream) {
  if (!ws) return K3MOE_E_WORKSPACE;
  if (misaligned(ws)) return K3MOE_E_ALIGN;
  wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<uint32_t*>(ws));
  return cudaGetLastError() == cudaSuccess ? K3MOE_OK : K3MOE_E_CUDA;
}

}  // extern "C"

namespace k3moe {
namespace {
// One thread per CTA waits on the wall clock until `ns` nanoseconds have passed and returns; the
// CTA's dynamic shared memory (most of an SM's) keeps other large-shared-memory CTAs off its SM.
__global__ void occupy_kernel(unsigned long long ns) {
  extern __shared__ uint8_t occupy_smem[];
  if (threadIdx.x != 0) return;
  const unsigned long long t0 = globaltimer_ns();
  while (globaltimer_ns() - t0 < ns) __nanosleep(100000);
  occupy_smem[0] = 0;
}
constexpr size_t kOccupySmem = 200 * 1024;
}  // namespace
}  // namespace k3moe

extern "C" {

k3moe_status k3moe_selftest_occupy(int32_t n_ctas, int32_t ms, void* stream) {
  if (n_ctas < 1 || n_ctas > 4096 || ms < 1 || ms > 10000) return K3MOE_E_SHAPE;
  if (ensure_smem_attr(reinterpret_cast<const void*>(occupy_kernel), kOccupySmem) != cudaSuccess)
    return K3MOE_E_CUDA;
  occupy_kernel<<<n_ctas, 32, kOccupySmem, static_cast<cudaStream_t>(stream)>>>(1000000ull * (unsigned)ms);
  return cudaGetLastError() == cudaSuccess ? K3MOE_OK : K3MOE_E_CUDA;
}

k3moe_status k3moe_check(void* ws, void* stream) {
  if (!ws) return K3MOE_E_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return K3MOE_E_CUDA;
  uint32_t word = 0;
  if (cudaMemcpy(&word, ws, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return K3MOE_E_CUDA;
  if (word != 0) {
    if (cudaMemset(ws, 0, sizeof(word)) != cudaSuccess) return K3MOE_E_CUDA;
    return (word & kErrTimeout) ? K3MOE_E_TIMEOUT : K3MOE_E_DEVICE;
  }
  return K3MOE_OK;
}

}  // extern "C"
