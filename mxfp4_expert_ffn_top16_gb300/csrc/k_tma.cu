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
  uint64_t inner, rows, pitch, chunks;  // chunks == 0: 2-D map
  uint32_t box_inner, box_rows, box_chunks, elem, swz;
  bool operator==(const Key& o) const { return std::memcmp(this, &o, sizeof(Key)) == 0; }
};

struct Entry {
  Key key;
  CUtensorMap map;
  bool used;
};

constexpr uint32_t kElemFp4 = 0x41;
constexpr int kCache = 64;
Entry g_cache[kCache];
int g_next = 0;
std::mutex g_mu;

bool encode_cached(CUtensorMap* out, const Key& k) {
  std::lock_guard<std::mutex> lock(g_mu);
  for (int i = 0; i < kCache; ++i)
    if (g_cache[i].used && g_cache[i].key == k) {
      *out = g_cache[i].map;
      return true;
    }
  auto enc = get_encode();
  if (!enc) return false;
  const int rank = k.chunks ? 3 : 2;
  // dim 0: `inner` contiguous elements; dim 1: rows `pitch` bytes apart; dim 2 (3-D only):
  // consecutive chunks of `inner` elements along a row (inner * elem bytes apart)
  cuuint64_t dims[3] = {k.inner, k.rows, k.chunks};
  // (an e2m1 chunk of `inner` codes takes inner / 2 bytes)
  cuuint64_t strides[2] = {k.pitch, k.elem == kElemFp4 ? (cuuint64_t)k.inner / 2 : (cuuint64_t)k.inner * k.elem};
  cuuint32_t box[3] = {k.box_inner, k.box_rows, k.box_chunks};
  cuuint32_t estr[3] = {1, 1, 1};
  CUtensorMap m;
  // elem 1: bytes; 2: bf16; kElemFp4: e2m1 pairs, 16 codes (8 bytes) per 16-byte unit in shared memory
  const CUtensorMapDataType dt = k.elem == 1   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : k.elem == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                               : CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B;
  const CUresult r = enc(&m, dt,
                         (cuuint32_t)rank, const_cast<void*>(k.base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE,
                         k.swz ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
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
  return encode_cached(out, k);
}

bool make_tmap_fp4(CUtensorMap* out, const void* base, uint64_t inner, uint64_t rows, uint64_t pitch_bytes,
                   uint32_t box_rows) {
  Key k;
  std::memset(&k, 0, sizeof(k));
  k.base = base;
  k.inner = inner;
  k.rows = rows;
  k.pitch = pitch_bytes;
  k.box_inner = 128;
  k.box_rows = box_rows;
  k.elem = kElemFp4;
  k.swz = 1u;
  return encode_cached(out, k);
}

bool make_tmap_3d_chunks(CUtensorMap* out, const void* base, int elem_bytes, uint64_t chunk, uint64_t rows,
                         uint64_t pitch_bytes, uint64_t nchunks, uint32_t box_rows, uint32_t box_chunks,
                         bool swizzle128) {
  Key k;
  std::memset(&k, 0, sizeof(k));
  k.base = base;
  k.inner = chunk;
  k.rows = rows;
  k.pitch = pitch_bytes;
  k.chunks = nchunks;
  k.box_inner = (uint32_t)chunk;
  k.box_rows = box_rows;
  k.box_chunks = box_chunks;
  k.elem = (uint32_t)elem_bytes;
  k.swz = swizzle128 ? 1u : 0u;
  return encode_cached(out, k);
}

bool make_tmap_fp4_chunks(CUtensorMap* out, const void* base, uint64_t inner, uint64_t rows, uint64_t pitch_bytes,
                          uint32_t box_rows, uint32_t box_chunks) {
  Key k;
  std::memset(&k, 0, sizeof(k));
  k.base = base;
  k.inner = 128;
  k.rows = rows;
  k.pitch = pitch_bytes;
  k.chunks = inner / 128;
  k.box_inner = 128;
  k.box_rows = box_rows;
  k.box_chunks = box_chunks;
  k.elem = kElemFp4;
  k.swz = 1u;
  return encode_cached(out, k);
}

}  // namespace k3moe
