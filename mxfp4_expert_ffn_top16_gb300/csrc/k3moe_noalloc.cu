// k3moe_route_noalloc: router logits + top-k with no workspace from the caller and no device
// allocation. The logits live in one fixed scratch array that is part of the library's own
// device image, so every GPU that loads the library holds it until the process exits.
//
// Host code must not hand the symbol g_route_scratch itself to a kernel: on the host that name
// is only a stand-in, not a device address. The device address comes from
// cudaGetSymbolAddress, looked up once per device (with that device current) on the first call
// made on it, and cached.
#include <mutex>

#include <cuda_runtime.h>

#include "k3moe_internal.cuh"

namespace k3moe {
namespace {

// Error word (first 256 bytes), then router logits, fp32, [T][E] with T * E <= kMaxLogits.
constexpr size_t kHeaderBytes = 256;
constexpr size_t kMaxLogits = 65536;
constexpr size_t kScratchBytes = kHeaderBytes + kMaxLogits * sizeof(float);  // 262,400 bytes

static __device__ __align__(256) unsigned char g_route_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of g_route_scratch on the current device; the first call per device looks it up.
k3moe_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return K3MOE_E_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return K3MOE_E_DEVICE;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || !p) return K3MOE_E_CUDA;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return K3MOE_OK;
}

bool misaligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

}  // namespace
}  // namespace k3moe

using namespace k3moe;

extern "C" k3moe_status k3moe_route_noalloc(const k3moe_dims* dims, const uint16_t* x, int32_t T,
                                            const uint16_t* w_router, const float* bias, int32_t* topk_idx,
                                            float* topk_w, uint32_t* err_word, void* stream) {
  size_t unused = 0;
  const k3moe_status sd = k3moe_workspace_size(dims, 0, &unused);  // checks dims, allocates nothing
  if (sd != K3MOE_OK) return sd;
  const k3moe_dims& d = *dims;
  if (T < 0) return K3MOE_E_SHAPE;
  if ((size_t)T * (size_t)d.n_experts > kMaxLogits) return K3MOE_E_SCRATCH;
  if (!x || !w_router || !topk_idx || !topk_w) return K3MOE_E_NULL;
  if (misaligned16(x) || misaligned16(w_router) || misaligned16(bias) || misaligned16(topk_idx) ||
      misaligned16(topk_w) || misaligned16(err_word))
    return K3MOE_E_ALIGN;
  void* scratch = nullptr;
  const k3moe_status sa = scratch_address(&scratch);
  if (sa != K3MOE_OK) return sa;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t* err = err_word ? err_word : static_cast<uint32_t*>(scratch);
  // the error word must start at zero; the logits are fully rewritten before they are read
  if (cudaMemsetAsync(err, 0, sizeof(uint32_t), s) != cudaSuccess) return K3MOE_E_CUDA;
  if (T == 0) return K3MOE_OK;
  float* logits = reinterpret_cast<float*>(static_cast<unsigned char*>(scratch) + kHeaderBytes);
  if (launch_dense(w_router, d.n_experts, logits, nullptr, bias, nullptr, 0, nullptr, nullptr, nullptr, 0, x, T,
                   d.hidden, err, s) != cudaSuccess)
    return K3MOE_E_CUDA;
  if (launch_topk(logits, T, d.n_experts, d.top_k, topk_idx, topk_w, s) != cudaSuccess) return K3MOE_E_CUDA;
  return K3MOE_OK;
}
