// Host side of the TMA tiled copies: 2-D tensor maps over row-major global arrays, encoded
// through the driver entry point that the CUDA runtime exposes (no link-time dependency on
// the driver library) and cached by (address, shape, box, swizzle), so repeated calls on the
// same weights pay the encoding once.
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "k3moe_internal.cuh"

namespace k3moe {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

struct Key {
  const void* base;
  uint64_t inner, rows, pitch;
  uint32_t box_inner, box_rows, elem, swz;
  bool operator==(const Key& o) const { return std::memcmp(this, &o, sizeof(Key)) == 0; }
};

struct Entry {
  Key key;
  CUtensorMap map;
  bool used;
};

constexpr int kCache = 64;
Entry g_cache[kCache];
int g_next = 0;
std::mutex g_mu;

}  // namespace

bool make_tmap_2d(CUtensorMap* out, const void* base, int elem_bytes, uint64_t inner, uint64_t rows,
                  uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_rows, bool swizzle128) {
  Key k;
  std::memset(&k, 0, sizeof(k));
  k.base = base;
  k.inner = inner;
  k.rows = rows;
  k.pitch = pitch_bytes;
  k.box_inner = box_inner;
  k.box_rows = box_rows;
  k.elem = (uint32_t)elem_bytes;
  k.swz = swizzle128 ? 1u : 0u;
  std::lock_guard<std::mutex> lock(g_mu);
  for (int i = 0; i < kCache; ++i)
    if (g_cache[i].used && g_cache[i].key == k) {
      *out = g_cache[i].map;
      return true;
    }
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {pitch_bytes};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUtensorMap m;
  const CUresult r = enc(&m, elem_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                         const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  Entry& e = g_cache[g_next];
  g_next = (g_next + 1) % kCache;
  e.key = k;
  e.map = m;
  e.used = true;
  *out = m;
  return true;
}

}  // namespace k3moe
