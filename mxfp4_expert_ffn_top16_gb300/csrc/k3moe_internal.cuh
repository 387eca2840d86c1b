// Internal declarations shared by the libk3moe translation units: workspace layout, the
// device error word, PTX wrappers (mbarrier, bulk copy, mma.sync, format conversions) and
// the kernel launchers. Not part of the public interface (include/k3moe.h is).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "k3moe.h"

namespace k3moe {

// ------------------------------------------------------------------ error word
// Bits of the uint32 error word at offset 0 of the workspace.
constexpr uint32_t kErrTimeout = 1u;   // a bounded mbarrier wait ran out
constexpr uint32_t kErrIndex = 2u;     // a device-side index check failed

// Wall-clock bound of every device-side wait, in nanoseconds (%globaltimer).
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// ------------------------------------------------------------------ workspace layout
struct WsLayout {
  size_t err, logits, idx, wts, offsets, row_token, row_slot, slot_row;
  size_t plan;          // int32: [0] n_active, [1] total chunks, [2..] active ids, chunk prefix
  size_t z, zh, zs;     // latent activations: bf16, f16 block-scaled copy, block exponents
  size_t a, ah, as;     // GLU output per sorted row: bf16, f16 block-scaled copy, exponents
  size_t o;             // fp32 expert outputs per sorted row
  size_t c;             // bf16 combined latent
  size_t perm;          // int32 per-block histograms of the multi-block permutation
  size_t total;
};
WsLayout ws_layout(const k3moe_dims& d, int64_t T);

// Tokens per column tile of the expert GEMV (one mma.m16n8 n-tile).
constexpr int kGemvTokens = 8;
// Features per unit of the expert GEMV and of the dense GEMV.
constexpr int kUnitRows = 32;

// Plan: active experts and their token chunks, used to schedule the expert GEMV.
//   plan[0] = number of active experts D, plan[1] = total chunks C,
//   plan[2 .. 2+E)        = active expert ids (first D valid),
//   plan[2+E .. 2+2E+1)   = chunk prefix over active experts (first D+1 valid).
inline size_t plan_ints(int E) { return 2 + 2 * (size_t)E + 1; }

// ------------------------------------------------------------------ launchers
// Each returns cudaSuccess or the launch error.
cudaError_t launch_dense_gemv(const uint16_t* W0, int N0, float* out0_f32, uint16_t* out0_bf16,
                              const float* bias0, const uint16_t* W1, int N1, uint16_t* out1_bf16,
                              __half* out1_h, int8_t* out1_s, int actq1, const uint16_t* x, int T,
                              int K, uint32_t* err, cudaStream_t s);
cudaError_t launch_topk(const float* logits, int T, int E, int k, int32_t* idx, float* w,
                        cudaStream_t s);
cudaError_t launch_permute(const int32_t* idx, int T, int E, int k, int32_t* offsets,
                           int32_t* row_token, int32_t* row_slot, int32_t* slot_row,
                           int32_t* plan, int32_t* scratch, uint32_t* err, cudaStream_t s);
cudaError_t launch_plan(const int32_t* offsets, int E, int32_t* plan, cudaStream_t s);
cudaError_t launch_act_prep(const uint16_t* z, int T, int L, int actq, __half* zh, int8_t* zs,
                            cudaStream_t s);
cudaError_t launch_expert_glu(const k3moe_dims& d, const k3moe_weights& w, const int32_t* plan,
                              const int32_t* offsets, const int32_t* row_token, const __half* zh,
                              const int8_t* zs, uint16_t* a, __half* ah, int8_t* as, int rows_max,
                              uint32_t* err, cudaStream_t s);
cudaError_t launch_expert_down(const k3moe_dims& d, const k3moe_weights& w, const int32_t* plan,
                               const int32_t* offsets, const __half* ah, const int8_t* as,
                               float* o_rows, int rows_max, uint32_t* err, cudaStream_t s);
cudaError_t launch_combine(const float* o_rows, const int32_t* slot_row, const float* w, int T,
                           int k, int L, uint16_t* c, cudaStream_t s);

int num_sms();

}  // namespace k3moe
