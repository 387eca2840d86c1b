// Device-side helpers for libk3moe kernels: number formats, mbarrier waits with a wall-clock
// bound, bulk copies (TMA engine), legacy mma.sync tiles and warp reductions.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "k3moe_internal.cuh"

namespace k3moe {

// ------------------------------------------------------------------ number formats
__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// fp32 -> bf16, round to nearest even (NaN stays NaN).
__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40u);
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

// One term of the routing-weighted combine: s += w * v as a Kahan-compensated fp32 sum (c the
// compensation), the product rounded on its own. Explicit round-to-nearest operations, so the
// product is never contracted into the sum and the result does not depend on the compiler.
__device__ __forceinline__ void combine_term(float& s, float& c, float w, float v) {
  const float y = __fsub_rn(__fmul_rn(w, v), c);
  const float t = __fadd_rn(s, y);
  c = __fsub_rn(__fsub_rn(t, s), y);
  s = t;
}
__device__ __forceinline__ uint16_t combine_result(float s, float c) { return f32_to_bf16(__fsub_rn(s, c)); }

// floor(log2|v|) for a finite nonzero normal fp32 v; -127 for zero and subnormals.
__device__ __forceinline__ int ilog2_floor(float v) {
  int e = (int)((__float_as_uint(v) >> 23) & 0xff);
  return e == 0 ? -127 : e - 127;
}

// 2^e as fp32 for e in [-126, 127].
__device__ __forceinline__ float exp2i(int e) { return __uint_as_float((uint32_t)(e + 127) << 23); }

// e8m0 byte -> fp32 scale 2^(E-127). E = 0 flushes to 0; E = 255 gives +inf.
__device__ __forceinline__ float e8m0_to_f32(uint32_t E) { return __uint_as_float(E << 23); }

// MXFP8 round trip of one value given its block's shared exponent X (OCP MX v1.0):
// v / 2^X rounded to E4M3 (nearest even, saturating at 448), then scaled back by 2^X.
__device__ __forceinline__ float mxfp8_roundtrip(float v, int X) {
  float s = ldexpf(v, -X);  // exact power-of-two scaling
  uint16_t pair;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pair) : "f"(0.0f), "f"(s));
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(pair));
  float q = __half2float(__ushort_as_half((uint16_t)(h2 & 0xffff)));
  return ldexpf(q, X);
}

// Shared exponent of an MXFP8 block from its amax: floor(log2 amax) - 8, clamped to
// [-127, 127]; an all-zero block gets -127.
__device__ __forceinline__ int mxfp8_block_exp(float amax) {
  if (!(amax > 0.0f)) return -127;
  if (!(amax <= 3.4028235e38f)) return 127;
  int X = ilog2_floor(amax) - 8;
  return X < -127 ? -127 : (X > 127 ? 127 : X);
}

// Two values -> two E4M3 codes (nearest even, saturating), v0 in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float v0, float v1) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(v1), "f"(v0));
  return r;
}
// Two E4M3 codes (low byte first) -> their values.
__device__ __forceinline__ float2 e4m3x2_value(uint32_t pair) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)pair));
  return __half22float2(*reinterpret_cast<__half2*>(&h2));
}
// v * 2^e for e in [-254, 254] in two exact power-of-two steps.
__device__ __forceinline__ float mul_pow2(float v, int e) {
  const int e1 = e / 2;
  return v * exp2i(e1) * exp2i(e - e1);
}
// Block exponent of the hi / lo parts of a bf16 value split into two E4M3 rows
// (amax / 2^X in [128, 256)); all-zero block: -127.
__device__ __forceinline__ int split_block_exp(float amax) {
  if (!(amax > 0.0f)) return -127;
  if (!(amax <= 3.4028235e38f)) return 127;
  const int X = ilog2_floor(amax) - 7;
  return X < -127 ? -127 : (X > 127 ? 127 : X);
}
// Exponent of the first E4M3 row of a block: P = 1 MXFP8, P = 2 the hi part of the split.
template <int P>
__device__ __forceinline__ int block_exp(float amax) {
  return P == 1 ? mxfp8_block_exp(amax) : split_block_exp(amax);
}

// f16 block exponent: the power of two that brings a block's amax into [2^14, 2^15).
__device__ __forceinline__ int f16_block_exp(float amax) {
  if (!(amax > 0.0f) || !(amax <= 3.4028235e38f)) return 0;
  int e = ilog2_floor(amax) - 14;
  return e < -100 ? -100 : (e > 100 ? 100 : e);
}

// ------------------------------------------------------------------ programmatic dependent launch
// Kernels of the layer chain are launched so that the next one may start its prologue while
// this one finishes. pdl_wait() blocks until the preceding grid has completed and its writes
// are visible; every kernel calls it before its first global memory access. pdl_trigger()
// lets the following grid launch. Both are no-ops for a normal launch.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ------------------------------------------------------------------ warp reductions
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// ------------------------------------------------------------------ shared memory, mbarrier
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Waits for phase `parity` of `bar`. Gives up when *abort becomes nonzero (another thread
// gave up) or after kWaitLimitNs of wall time, in which case it records kErrTimeout in the
// error word, raises *abort and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  volatile int* abort, uint32_t* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 63u) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs || i > 0x7fffffffu) {
        *abort = 1;
        atomicOr(err, 1u);
        return false;
      }
    }
  }
}

// 1-D bulk copy global -> shared through the TMA engine; completion counted on `bar` as
// transaction bytes. dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// 2-D tiled copy global -> shared (TMA): the box at (x, y) of the tensor map lands at dst
// (1024-byte aligned for the 128-byte swizzle); completion counted on `bar` in bytes (out of
// range parts of the box are zero-filled and still counted). x * element size must be a
// multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

// Streaming loads of weights that are read once per step: an L2 policy that evicts them first,
// so that what the next kernels read again (their code, the small activation and routing
// tensors) is not pushed out of L2 by hundreds of MB of weights.
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void tma_load_3d_stream(void* dst, const CUtensorMap* map, int x, int y, int z,
                                                   uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
      "%3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void tma_load_2d_stream(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                                   uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
      "%3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void bulk_g2s_stream(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                                uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Byte offset of (row r, byte c) inside a box whose rows are 128 bytes and which was written
// with the 128-byte swizzle: the 16-byte chunk index is XORed with r mod 8.
__device__ __forceinline__ int swz128(int r, int c) {
  return r * 128 + ((((c >> 4) ^ r) & 7) << 4) + (c & 15);
}

// ------------------------------------------------------------------ mma.sync tiles
// D(16x8 f32) += A(16x16 f16, row) * B(16x8 f16, col)
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// D(16x8 f32) += A(16x16 bf16, row) * B(16x8 bf16, col)
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two e2m1 codes (one byte, weight 2j in the low nibble) -> f16x2 (low half = weight 2j).
// The hardware conversion applies the 16-entry e2m1 value table.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t r;
  asm("{ .reg .b8 t; cvt.u8.u32 t, %1; cvt.rn.f16x2.e2m1x2 %0, t; }" : "=r"(r) : "r"(byte));
  return r;
}

// Four bytes of codes (8 weights, low nibble first) -> four f16x2 registers, byte j -> r[j].
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t (&r)[4]) {
  asm("{ .reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3; }"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "r"(w));
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Bounded wait by a whole warp: lane 0 polls, the result goes to every lane, and the warp
// synchronises, so the lanes never part ways on a timeout and all see what lane 0 acquired.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, volatile int* abort,
                                               uint32_t* err) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait_bounded(bar, parity, abort, err);
  ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  __syncwarp();
  return ok;
}

// Barrier over a fixed group of warps (the mbarrier's arrival count = number of warps; lane 0
// of each warp arrives after the warp synchronises), with the same bounded wait as the
// pipeline barriers, so a group member that gave up cannot strand the others. `phase` is the
// caller's running parity for this barrier. Call with the whole warp.
__device__ __forceinline__ bool group_barrier(uint64_t* bar, uint32_t& phase, volatile int* abort,
                                              uint32_t* err) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
  const bool ok = mbar_wait_bounded(bar, phase, abort, err);
  phase ^= 1u;
  return ok;
}

// group_barrier with a warp-wide wait (mbar_wait_warp): every lane leaves with the same result.
__device__ __forceinline__ bool group_barrier_warp(uint64_t* bar, uint32_t& phase, volatile int* abort,
                                                   uint32_t* err) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
  const bool ok = mbar_wait_warp(bar, phase, abort, err);
  phase ^= 1u;
  return ok;
}

}  // namespace k3moe
