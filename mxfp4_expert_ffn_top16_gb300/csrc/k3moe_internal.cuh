// Internal declarations shared by the libk3moe translation units: workspace layout, the
// device error word, PTX wrappers (mbarrier, bulk copy, mma.sync, format conversions) and
// the kernel launchers. Not part of the public interface (include/k3moe.h is).
#pragma once

#include <cstddef>
#include <cstdint>
#include <utility>
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "k3moe.h"

namespace k3moe {

// 2-D tensor map over a row-major array: `inner` elements per row (contiguous), `rows` rows
// `pitch_bytes` apart, box of box_inner x box_rows elements, optional 128-byte swizzle.
// Cached by its arguments. Returns false if the driver entry point or the encoding fails.
bool make_tmap_2d(CUtensorMap* out, const void* base, int elem_bytes, uint64_t inner, uint64_t rows,
                  uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_rows, bool swizzle128);
// 3-D view of a row-major [rows][nchunks * chunk] array as {chunk, rows, nchunks}: one box of
// {chunk, box_rows, box_chunks} lands as box_chunks consecutive [box_rows][chunk] tiles, so a
// single copy fetches several K-tiles of the same rows.
bool make_tmap_3d_chunks(CUtensorMap* out, const void* base, int elem_bytes, uint64_t chunk, uint64_t rows,
                         uint64_t pitch_bytes, uint64_t nchunks, uint32_t box_rows, uint32_t box_chunks,
                         bool swizzle128);
// Packed e2m1 codes, `inner` 4-bit codes per row `pitch_bytes` apart (16U4_ALIGN16B): a box of
// 128 codes x box_rows rows lands as box_rows rows of 128 bytes (each 8 bytes of codes padded to
// 16), 128-byte swizzle; the copy counts inner/2 bytes per row. `inner` and the pitch must be
// multiples of 128 codes and 16 bytes.
bool make_tmap_fp4(CUtensorMap* out, const void* base, uint64_t inner, uint64_t rows, uint64_t pitch_bytes,
                   uint32_t box_rows);
// e2m1 codes [rows][inner] as 3-D {128 codes, rows, inner / 128 chunks} (inner a multiple of
// 128): a box of box_rows rows x box_chunks consecutive 128-code chunks, each chunk a 128-byte
// swizzled tile of box_rows rows in shared memory.
bool make_tmap_fp4_chunks(CUtensorMap* out, const void* base, uint64_t inner, uint64_t rows, uint64_t pitch_bytes,
                          uint32_t box_rows, uint32_t box_chunks);

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
  size_t route_done;    // int in the header: top-k blocks finished (a few tokens); back to zero after each launch
  size_t sg, su, sa;    // shared experts: gate, up (fp32) and GLU output (bf16) [T][S]
  // block-scaled tensor-core expert path (only when umma_expert_ok): per sorted row, P e4m3
  // rows of z and of the GLU output with e8m0 scales per 32 (row pitch exp_pitch bytes)
  size_t bq, bs, aq, aqs;
  size_t chunk_done;    // int per chunk: GLU items finished (decode kernel running both passes)
  size_t xin, yout;     // k3moe_layer_run_host: the tokens and the output on the device [T][H] bf16
  size_t total;
};
WsLayout ws_layout(const k3moe_dims& d, int64_t T);

// Tokens per column tile of the expert GEMV (one mma.m16n8 n-tile).
constexpr int kGemvTokens = 8;
// Row pitch in bytes of the per-32-block exponent arrays of the f16 activation copies
// (K/32 bytes rounded up to 16 so rows can be bulk-copied).
inline __host__ __device__ int exp_pitch(int K) { return ((K / 32) + 15) & ~15; }
// Features per unit of the expert GEMV and of the dense GEMV.
constexpr int kUnitRows = 32;

// Plan: active experts and their token chunks, used to schedule the expert GEMV.
//   plan[0] = number of active experts D, plan[1] = total chunks C,
//   plan[2 .. 2+E)        = active expert ids (first D valid),
//   plan[2+E .. 2+2E+1)   = chunk prefix over active experts (first D+1 valid).
inline __host__ __device__ size_t plan_ints(int E) { return 2 + 2 * (size_t)E + 1; }
// The chunk table follows the plan ints: int4 {expert, first sorted row, rows, 0} per chunk of
// up to kGemvTokens rows, for at most rows/kGemvTokens + E chunks.
inline __host__ __device__ size_t plan_ctab_offset(int E) { return (plan_ints(E) * 4 + 15) & ~(size_t)15; }
inline __host__ __device__ int4* plan_ctab(int32_t* plan, int E) {
  return reinterpret_cast<int4*>(reinterpret_cast<char*>(plan) + plan_ctab_offset(E));
}
// A second table for the tensor-core expert GEMM follows: entry 0 = {chunks C64, chunks of the
// experts with more than kSmallExpertRows rows, 0, 0}, entries 1..C64 = {expert, first sorted
// row, rows, 0}: first those experts' chunks of up to kUmmaChunkRows rows, then the other
// experts' chunks of up to kGemvTokens rows.
constexpr int kUmmaChunkRows = 112;
// With MXFP8 activations (one e4m3 row per sorted row) the chunks of the experts with more than
// kSmallExpertRows rows hold up to this many rows (the same MMA N and tile bytes as 112 rows of
// bf16 hi + lo pairs), so the big experts' weight tiles are streamed half as often.
constexpr int kUmmaChunkRowsWide = 224;
// With MXFP4 activations: 192 rows (a second 128-row block of activation scales then fits in
// tensor memory beside two accumulators).
constexpr int kUmmaChunkRowsFp4 = 192;
inline __host__ __device__ int many_chunk_rows(int actq) {
  return actq == 1 ? kUmmaChunkRowsWide : (actq == 2 ? kUmmaChunkRowsFp4 : kUmmaChunkRows);
}
// With many tokens the experts with at most this many sorted rows run on the weights-on-N
// decode kernel, in chunks of kGemvTokens rows (kSmallChunksMax at most per expert).
constexpr int kSmallExpertRows = kGemvTokens;
constexpr int kSmallChunksMax = (kSmallExpertRows + kGemvTokens - 1) / kGemvTokens;
// Bound on the entries of the second table.
inline __host__ __device__ long long plan_ctab64_max(int E, long long rows) {
  return rows / kUmmaChunkRows + (long long)E * kSmallChunksMax;
}
inline __host__ __device__ size_t plan_ctab64_offset(int E, long long rows) {
  return plan_ctab_offset(E) + (size_t)(rows / kGemvTokens + E + 1) * 16;
}
inline __host__ __device__ int4* plan_ctab64(int32_t* plan, int E, long long rows) {
  return reinterpret_cast<int4*>(reinterpret_cast<char*>(plan) + plan_ctab64_offset(E, rows));
}
inline __host__ __device__ size_t plan_bytes(int E, long long rows) {
  return plan_ctab64_offset(E, rows) + (size_t)(plan_ctab64_max(E, rows) + 2) * 16;
}

// ------------------------------------------------------------------ launchers
// Each returns cudaSuccess or the launch error.
// zero / nzero (optional): ints the kernel clears after its grid dependency wait (the decode
// expert kernel's counters, when no routing kernel runs in between).
cudaError_t launch_dense_gemv(const uint16_t* W0, int N0, float* out0_f32, uint16_t* out0_bf16,
                              const float* bias0, const uint16_t* W1, int N1, uint16_t* out1_bf16,
                              __half* out1_h, int8_t* out1_s, int actq1, const uint16_t* x, int T,
                              int K, uint32_t* err, cudaStream_t s, uint8_t* out1_q = nullptr,
                              uint8_t* out1_qs = nullptr, int q1P = 0, float* out1_f32 = nullptr,
                              const uint16_t* W0b = nullptr, const uint16_t* xb = nullptr, int Kb = 0,
                              int* zero = nullptr, int nzero = 0);
// Same contract as launch_dense_gemv (less the E4M3 rows), on tcgen05 tiles (for many tokens).
cudaError_t launch_umma_dense(const uint16_t* W0, int N0, float* out0_f32, uint16_t* out0_bf16,
                              const float* bias0, const uint16_t* W1, int N1, uint16_t* out1_bf16,
                              __half* out1_h, int8_t* out1_s, int actq1, const uint16_t* x, int T, int K,
                              uint32_t* err, cudaStream_t s, float* out1_f32 = nullptr,
                              const uint16_t* W0b = nullptr, const uint16_t* xb = nullptr, int Kb = 0);
// Token count from which the dense projections use the tcgen05 tiles.
constexpr int kUmmaDenseMinTokens = 33;
// out1_q / out1_qs / q1P (token-at-a-time path, T < kUmmaDenseMinTokens, only): problem 1's bf16
// outputs also as q1P E4M3 rows per token with e8m0 scales per 32, for the decode expert kernel.
// out1_f32: problem 1's sums in fp32. W0b / xb / Kb: a second K segment of problem 0 (with no
// problem 1): out0 = W0 x + W0b xb, W0b [N0][Kb], xb [T][Kb], one rounding of the total.
inline cudaError_t launch_dense(const uint16_t* W0, int N0, float* out0_f32, uint16_t* out0_bf16,
                                const float* bias0, const uint16_t* W1, int N1, uint16_t* out1_bf16,
                                __half* out1_h, int8_t* out1_s, int actq1, const uint16_t* x, int T, int K,
                                uint32_t* err, cudaStream_t s, uint8_t* out1_q = nullptr,
                                uint8_t* out1_qs = nullptr, int q1P = 0, float* out1_f32 = nullptr,
                                const uint16_t* W0b = nullptr, const uint16_t* xb = nullptr, int Kb = 0,
                                int* zero = nullptr, int nzero = 0) {
  if (T >= kUmmaDenseMinTokens)
    return launch_umma_dense(W0, N0, out0_f32, out0_bf16, bias0, W1, N1, out1_bf16, out1_h, out1_s, actq1, x,
                             T, K, err, s, out1_f32, W0b, xb, Kb);
  return launch_dense_gemv(W0, N0, out0_f32, out0_bf16, bias0, W1, N1, out1_bf16, out1_h, out1_s, actq1, x,
                           T, K, err, s, out1_q, out1_qs, q1P, out1_f32, W0b, xb, Kb, zero, nzero);
}
cudaError_t launch_topk(const float* logits, int T, int E, int k, int32_t* idx, float* w,
                        cudaStream_t s);
cudaError_t launch_permute(const int32_t* idx, int T, int E, int k, int32_t* offsets,
                           int32_t* row_token, int32_t* row_slot, int32_t* slot_row,
                           int32_t* plan, int32_t* scratch, uint32_t* err, cudaStream_t s,
                           int big_rows = kUmmaChunkRows);
// big_rows: rows per chunk of the experts with more than kSmallExpertRows rows in the plan's
// many-token chunk table (many_chunk_rows of the activation mode).
cudaError_t launch_plan(const int32_t* offsets, int E, int rows_max, int32_t* plan, uint32_t* err,
                        cudaStream_t s, int big_rows = kUmmaChunkRows);
// Top-k (one block per token), then permutation + plan in one block, for T <= kSmallRouteTokens.
constexpr int kSmallRouteTokens = 64;
// done: a workspace counter that is zero between launches (the workspace starts zeroed). Also
// clears the ncnt counters at cnt (the decode expert kernel's per-chunk GLU completion counts).
cudaError_t launch_route_tail_small(const float* logits, int T, int E, int k, int32_t* idx, float* w,
                                    int32_t* offsets, int32_t* row_token, int32_t* row_slot,
                                    int32_t* slot_row, int32_t* plan, int* done, int* cnt, int ncnt,
                                    uint32_t* err, cudaStream_t s);
cudaError_t launch_act_prep(const uint16_t* z, int T, int L, int actq, __half* zh, int8_t* zs,
                            cudaStream_t s);
cudaError_t launch_expert_glu(const k3moe_dims& d, const k3moe_weights& w, const int32_t* plan,
                              const int32_t* offsets, const int32_t* row_token, const __half* zh,
                              const int8_t* zs, uint16_t* a, __half* ah, int8_t* as, int T,
                              uint32_t* err, cudaStream_t s);
cudaError_t launch_expert_down(const k3moe_dims& d, const k3moe_weights& w, const int32_t* plan,
                               const int32_t* offsets, const __half* ah, const int8_t* as,
                               float* o_rows, int T, uint32_t* err, cudaStream_t s);
// Block-scaled tensor-core expert GEMMs. Usable when latent and inter are multiples of 128
// (otherwise the expert GEMV runs). P = 2 (bf16 activations as e4m3 hi + lo) or 1 (MXFP8
// activations). Items are chunks of up to kUmmaChunkRows sorted rows from
// kUmmaExpertMinTokens tokens on, of up to kGemvTokens rows below.
constexpr int kUmmaExpertMinTokens = 65;
inline bool umma_expert_ok(const k3moe_dims& d) { return d.latent % 128 == 0 && d.inter % 128 == 0; }
// Rows per chunk of the tensor-core expert kernels: P activation rows per sorted row (0: MXFP4).
inline int umma_chunk_rows(long long T, int P) {
  return T < kUmmaExpertMinTokens ? kGemvTokens
                                  : (P == 1 ? kUmmaChunkRowsWide : (P == 0 ? kUmmaChunkRowsFp4 : kUmmaChunkRows));
}
// z rows gathered by row_token into P e4m3 rows per sorted row: bq [P*rows][L], bs [P*rows][exp_pitch(L)]
// (row_token null: row r is token r). Also clears the ncnt counters at cnt (the decode kernel's
// per-chunk GLU completion counts).
// slot_row (optional, with k): convert each token once and store it to the sorted rows of its k
// slots (rows = T * k) instead of converting every sorted row from its token.
cudaError_t launch_quant_rows(const uint16_t* z, const int32_t* row_token, int rows, int T, int L, int P,
                              uint8_t* bq, uint8_t* bs, int* cnt, int ncnt, uint32_t* err, cudaStream_t s,
                              const int32_t* slot_row = nullptr, int k = 0);
// big_only (many tokens): only the chunks of the experts with more than kSmallExpertRows rows
// (the others then go to launch_umma_wn with small_experts).
// ps (may be null): the weight scales from the prepared layer's staging images, one bulk copy
// per stage instead of a gather per weight row.
struct PackedScales;
cudaError_t launch_umma_glu(const k3moe_dims& d, const k3moe_weights& w, int32_t* plan, const uint8_t* bq,
                            const uint8_t* bs, int P, int T, uint8_t* aq, uint8_t* aqs, uint32_t* err,
                            cudaStream_t s, bool big_only = false, const PackedScales* ps = nullptr);
cudaError_t launch_umma_down(const k3moe_dims& d, const k3moe_weights& w, int32_t* plan, const uint8_t* aq,
                             const uint8_t* aqs, int P, int T, float* o_rows, uint32_t* err, cudaStream_t s,
                             bool big_only = false, const PackedScales* ps = nullptr);
// Decode (T < kUmmaExpertMinTokens): both GEMMs in one launch, the weights on the MMA's M side
// (128 weight rows per MMA) and a chunk's up to 8 sorted rows on N. chunk_done: decode_counters
// ints, zero at launch (GLU items finished per chunk, then the kernel's item counter); the kernel
// leaves them non-zero, the next routing or row-quantisation launch clears them.
// zq / zqs: the latent activations as P E4M3 rows per token [T][P][L] with e8m0 scales
// [T][P][exp_pitch(L)]; the kernel gathers a chunk's rows through row_token.
// ps (may be null): the weight scales repacked by launch_pack_scales.
struct PackedScales {
  const uint8_t* gate;  // gate_s, rows E * I, K = L
  const uint8_t* up;    // up_s
  const uint8_t* down;  // down_s, rows E * L, K = I
  const uint8_t* glu;   // gate_s and up_s interleaved per 64 features (launch_pack_scales_glu)
};
// Share of the latent-out weight the one-token expert kernel fetches into L2 while it selects
// the experts (the memory is otherwise idle then). Measured at one token: 0.25 -1.3 us per
// step, 0.35 -1.4 us, 0.5 -0.7 us, all of it -0.2 us (more of it competes with the expert
// weights' stream; the latent-out GEMV is not bound by HBM alone).
constexpr double kL2NextFraction = 0.35;
// sel (optional, one token): the kernel selects the experts itself from the router logits (no
// routing kernel before it); every CTA builds the plan in shared memory, CTA 0 also writes the
// routing outputs (topk_idx, topk_w, offsets, row_token, row_slot, slot_row, plan).
struct DecodeSelect {
  const float* logits;
  int32_t* idx;
  float* wts;
  int32_t* offsets;
  int32_t* row_token;
  int32_t* row_slot;
  int32_t* slot_row;
  // Optional: bytes [0, l2_next_bytes) of a weight the next kernel of the step reads (the
  // latent-out projection), fetched into L2 while the selection runs and the memory is idle.
  const void* l2_next;
  long long l2_next_bytes;
};
cudaError_t launch_umma_decode(const k3moe_dims& d, const k3moe_weights& w, const PackedScales* ps, int32_t* plan,
                               const uint8_t* zq, const uint8_t* zqs, const int32_t* row_token, int P, int T,
                               uint8_t* aq, uint8_t* aqs, float* o_rows, int* chunk_done, uint32_t* err,
                               cudaStream_t s, const DecodeSelect* sel = nullptr);
// The same GEMMs with the weights on the MMA's N side (256 weight rows per MMA, the chunk's
// activation rows on M = 128): half the MMA instructions per weight byte, which pays once chunks
// carry more than 8 activation rows. GLU pass, and with_down (latent % 256 == 0) the down pass in
// the same launch; chunk_done and zq / zqs as for launch_umma_decode.
// small_experts (many tokens): the chunks are those of the experts with at most
// kSmallExpertRows rows (the tail of the many-token chunk table), row_token is null and zq / zqs
// hold P rows per sorted row (the many-token quantised rows).
cudaError_t launch_umma_wn(const k3moe_dims& d, const k3moe_weights& w, const PackedScales* ps, int32_t* plan,
                           const uint8_t* zq, const uint8_t* zqs, const int32_t* row_token, int P, int T,
                           uint8_t* aq, uint8_t* aqs, bool with_down, float* o_rows, int* chunk_done,
                           uint32_t* err, cudaStream_t s, bool small_experts = false);
// Which decode kernel: the weights on M for bf16 activations (P = 2) with at most 4 tokens (a
// chunk then carries at most 8 activation rows) and for MXFP8 at one token, on N otherwise.
// Measured at decode_b1: 92.5 against 94.1 us per step for bf16, 92.6 against 91.8 for MXFP8
// before the one-token kernel selected its experts itself; with that (and the latent-out
// prefetch) MXFP8 takes 86.7 against 91.5 on the M side. At decode_b64 the N side is ahead in
// both modes.
inline bool decode_weights_on_m(int P, long long T) { return (P == 2 && T <= 4) || (P == 1 && T == 1); }
// e8m0 scales [rows][K/32] (rows a multiple of 128, K of 128) -> the decode kernel's staging
// image (same size): per 128 rows and 128-code chunk a 512-byte block whose byte 16 l + 4 w + q
// is the scale of row 32 w + l, K-block 4 chunk + q.
cudaError_t launch_pack_scales(const uint8_t* src, long long rows, int K, uint8_t* dst, cudaStream_t s);
// The gate and up scales (rows each, a multiple of 64) -> the many-token GLU tile's image (twice
// the size of one): per 64 features and 128-code chunk a 512-byte block whose byte 16 l + 4 w + q
// is the scale of tile row 32 w + l (rows 0..63 gate, 64..127 up of the same features).
cudaError_t launch_pack_scales_glu(const uint8_t* gate, const uint8_t* up, long long rows, int K, uint8_t* dst,
                                   cudaStream_t s);
inline int plan_chunks_max(const k3moe_dims& d, long long T) {
  return (int)(T * d.top_k / kGemvTokens + d.n_experts + 1);
}
// Counters of the decode expert kernel in the workspace: one per chunk, then its item counter.
inline int decode_counters(const k3moe_dims& d, long long T) { return plan_chunks_max(d, T) + 1; }
// a[i] = bf16(silu(g[i]) * u[i]) for n elements (the shared experts' GLU, fp32 in).
cudaError_t launch_glu(const float* g, const float* u, long long n, uint16_t* a, cudaStream_t s);
cudaError_t launch_combine(const float* o_rows, const int32_t* slot_row, const float* w, int T,
                           int k, int L, uint16_t* c, cudaStream_t s);
// dst[0, bytes) = src[0, bytes) with 16-byte loads and stores (either side may be page-locked host
// memory mapped into the device's address space); bytes a multiple of 16, both 16-byte aligned.
cudaError_t launch_copy16(const void* src, void* dst, size_t bytes, cudaStream_t s);
// S[idx[t][j]] += w[t][j] * ||o_rows[r]||_2 for every sorted row r of (t, j) (fp64 atomics).
cudaError_t launch_saliency(const float* o_rows, const int32_t* row_token, const int32_t* row_slot,
                            const int32_t* idx, const float* w, int T, int k, int L, int E, double* S,
                            uint32_t* err, cudaStream_t s);

int num_sms();

// Raises a kernel's dynamic shared-memory limit to at least `bytes` on the current device,
// calling the runtime only the first time (or when more is needed), so launches stay cheap.
cudaError_t ensure_smem_attr(const void* fn, size_t bytes);

// Launch with programmatic stream serialization (the kernel must call pdl_wait() before its
// first global memory access).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace k3moe
