/*
 * libk3moe -- one Stable-LatentMoE routed-expert layer with MXFP4 experts, on one GPU.
 *
 * The layer (Kimi K3, as the pages describe it):
 *   - "kimi-k3-mlx" digest, "Architecture" table: 896 routed experts, top-16 per token;
 *     the routed experts work in a 3584-wide latent space, not on the 7168-wide residual
 *     (Stable LatentMoE); the activation is a GLU evaluated in fp32.
 *   - "kimi-k3-in-c", "MXFP4 experts": expert weights are 4-bit codes indexing a 16-entry
 *     table, 32 consecutive weights share one 8-bit exponent, 17,547,264 bytes per expert.
 *   - "Kimi K3 hardware deep dive", quantisation-aware training: MXFP4 weights with MXFP8
 *     activations.
 *
 * Per token t (x_t in R^H, H = hidden):
 *   l      = W_r x_t + b                       router logits over E experts      (k3moe_route)
 *   S_t    = the k largest l (ties -> lowest index), reported in ascending index order
 *   w_j    = softmax(l)_j / sum_{i in S_t} softmax(l)_i, i.e. softmax over the kept logits
 *   z_t    = bf16(W_in x_t)                    latent in, [L][H]                 (k3moe_project)
 *   rows   = (token, slot) pairs grouped by expert, token order within an expert (k3moe_permute)
 *   o_tj   = D_e bf16(silu(G_e z_t) * (U_e z_t))  for e = S_t[j], MXFP4 G,U [I][L], D [L][I]
 *                                                                             (k3moe_expert_ffn_mxfp4)
 *   c_t    = bf16(sum_j w_j o_tj)              combine in latent space           (k3moe_combine)
 *   s_t    = sum_j D_j bf16(silu(G_j x_t) * (U_j x_t))   the n_shared always-on shared experts,
 *            bf16 G,U [Is][H], D [H][Is], on the residual ("kimi-k3-mlx", Architecture table:
 *            shared experts beside the routed ones, outside the latent space); 0 if none
 *   y_t    = bf16(W_out c_t + s_t)             latent out, [H][L], one rounding   (k3moe_project)
 * k3moe_layer_forward runs all of it. In MXFP8 mode (actq = 1) z and the GLU output go
 * through an MXFP8 round trip (E4M3 elements, one E8M0 scale per 32, OCP MX v1.0) before
 * they enter an expert matrix; in MXFP4 mode (actq = 2) through an MXFP4 round trip (E2M1
 * elements, one E8M0 scale per 32, OCP MX v1.0), and the experts run on the FP4 tensor rate
 * (the "Kimi K3 hardware deep dive", quantisation-aware training section, names MXFP4 weights
 * with MXFP8 activations; 4-bit activations are the mode the FP4 rate needs).
 *
 * Storage (all row-major, K contiguous; bf16 as uint16_t bit patterns):
 *   w_router [E][H] bf16, router_bias [E] fp32 (may be NULL), w_in [L][H], w_out [H][L] bf16.
 *   gate_q, up_q [E][I][L/2] uint8: two e2m1 codes per byte, weight 2j in the low nibble.
 *   gate_s, up_s [E][I][L/32] uint8: e8m0, value 2^(s-127), one per 32 weights along K.
 *   down_q [E][L][I/2], down_s [E][L][I/32] likewise.
 *
 * Conventions for every call:
 *   - Pointers are device pointers unless stated; the caller owns all memory (except the
 *     prepared-layer handle). No call allocates device memory or synchronises the stream
 *     (except k3moe_layer_init, k3moe_layer_free, k3moe_check and k3moe_layer_stats).
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *   - Work is enqueued asynchronously; a returned K3MOE_OK means the launches were accepted.
 *   - T = 0 is valid and does nothing.
 *   - Arguments are checked before anything is launched; a failed check launches nothing.
 *   - Device pointers must be 16-byte aligned (K3MOE_E_ALIGN otherwise).
 *   - hidden, latent and inter must be positive multiples of 64; 1 <= top_k <= 32,
 *     top_k <= n_experts <= 1024.
 *   - Faults the device detects (a bounded wait that ran out) are recorded in the
 *     workspace and reported by k3moe_check.
 *   - No call throws, exits or aborts.
 * Reported rather than guaranteed: e8m0 = 0 (2^-127) is flushed to zero by the expert
 * kernels, and e8m0 = 255 (NaN) makes the affected outputs non-finite.
 */
#ifndef K3MOE_H
#define K3MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum k3moe_status {
  K3MOE_OK = 0,
  K3MOE_E_NULL = 1,      /* a required pointer is NULL */
  K3MOE_E_SHAPE = 2,     /* a size is out of range or not a supported multiple */
  K3MOE_E_ALIGN = 3,     /* a device pointer is not 16-byte aligned */
  K3MOE_E_WORKSPACE = 4, /* workspace missing or smaller than k3moe_workspace_size() */
  K3MOE_E_MODE = 5,      /* act / actq not supported (act = 1, SiTU-GLU, has no formula; actq = 2
                            with latent or inter not a multiple of 256) */
  K3MOE_E_CUDA = 6,      /* a CUDA runtime call or launch failed */
  K3MOE_E_TIMEOUT = 7,   /* a device-side bounded wait ran out (see k3moe_check) */
  K3MOE_E_DEVICE = 8,    /* no usable sm_100-family device, or a device-side check failed */
  K3MOE_E_SCRATCH = 9,   /* request larger than k3moe_route_noalloc's fixed scratch */
  K3MOE_E_HOSTMEM = 10   /* a host buffer is not page-locked memory the device can address */
} k3moe_status;

typedef struct k3moe_dims {
  int32_t hidden;    /* H, residual width (K3: 7168) */
  int32_t latent;    /* L, latent width (K3: 3584) */
  int32_t inter;     /* I, expert intermediate width (K3: 3072) */
  int32_t n_experts; /* E (K3: 896) */
  int32_t top_k;     /* k (K3: 16) */
  int32_t act;       /* 0 = SiLU-GLU silu(gate) * up, fp32; 1 = SiTU-GLU -> K3MOE_E_MODE */
  int32_t actq;      /* 0 = bf16 activations; 1 = MXFP8 activations (E4M3 + E8M0 per 32);
                        2 = MXFP4 activations (E2M1 + E8M0 per 32; latent and inter multiples of 256) */
  int32_t n_shared;     /* always-on shared experts per token, 0..8 (K3: 2; 0 = none) */
  int32_t shared_inter; /* intermediate width of each shared expert (not on the pages; a
                           parameter); n_shared * shared_inter must be a multiple of 64 */
} k3moe_dims;

typedef struct k3moe_weights {
  const uint16_t* w_router;   /* [E][H] bf16 */
  const float* router_bias;   /* [E] fp32, added to the logits; may be NULL */
  const uint16_t* w_in;       /* [L][H] bf16 */
  const uint16_t* w_out;      /* [H][L] bf16 */
  const uint8_t* gate_q;      /* [E][I][L/2] */
  const uint8_t* gate_s;      /* [E][I][L/32] */
  const uint8_t* up_q;        /* [E][I][L/2] */
  const uint8_t* up_s;        /* [E][I][L/32] */
  const uint8_t* down_q;      /* [E][L][I/2] */
  const uint8_t* down_s;      /* [E][L][I/32] */
  /* Shared experts (used when n_shared > 0, else ignored), stacked: shared expert j owns rows
   * [j*Is, (j+1)*Is) of gate and up and the same columns of down (Is = shared_inter,
   * S = n_shared * Is). */
  const uint16_t* w_shared_gate; /* [S][H] bf16 */
  const uint16_t* w_shared_up;   /* [S][H] bf16 */
  const uint16_t* w_shared_down; /* [H][S] bf16 */
} k3moe_weights;

/* Bytes of device workspace that every call below needs for up to `max_tokens` tokens.
 * The workspace is caller-owned scratch; its first 256 bytes hold the device error word and a
 * counter the routing kernels return to zero after each launch. Zero it once after allocation
 * (cudaMemset); after that calls with any token count up to max_tokens may share it. */
k3moe_status k3moe_workspace_size(const k3moe_dims* dims, int32_t max_tokens, size_t* bytes);

/* Router scores and top-k ("kimi-k3-mlx", Architecture table: 896 experts, top-16).
 *   x [T][H] bf16, w_router [E][H] bf16, bias [E] fp32 or NULL.
 *   logits [T][E] fp32 out (may be NULL), topk_idx [T][k] int32 out (ascending expert
 *   index within a token), topk_w [T][k] fp32 out (renormalised softmax weights). */
k3moe_status k3moe_route(const k3moe_dims* dims, const uint16_t* x, int32_t T,
                         const uint16_t* w_router, const float* bias, float* logits,
                         int32_t* topk_idx, float* topk_w, void* ws, size_t ws_bytes,
                         void* stream);

/* k3moe_route without a workspace: the same router logits and top-k (same kernels, same
 * results as k3moe_route), with the logits kept in a fixed scratch array inside the library.
 * The pages have no counterpart; this exists for callers that cannot allocate device memory
 * for a routing decision: a serving process whose device memory is all handed to its own
 * pool allocator, where cudaMalloc / cudaFree are off limits on the request path because
 * they can synchronise the whole device and stall every other stream.
 *   x [T][H] bf16, w_router [E][H] bf16, bias [E] fp32 or NULL, topk_idx [T][k] int32 out,
 *   topk_w [T][k] fp32 out, as for k3moe_route.
 *   err_word: optional uint32 device output; cleared by this call, then set nonzero if the
 *   device detects a fault (a bounded wait that ran out). NULL keeps that word in the scratch.
 * Limit: T * n_experts <= 65536 (for 896 experts, up to 73 tokens); larger requests return
 * K3MOE_E_SCRATCH and launch nothing. The scratch is 262,400 bytes, part of the library's
 * device image, held on every GPU that loads the library until the process exits.
 * Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 * The first call on a device looks up the scratch's device address (once, with that device
 * current); make that first call before any stream capture. All calls share the one scratch
 * array: calls whose work can overlap on the GPU (different streams, or several host threads)
 * race on it and must be ordered by the caller. The looked-up address is kept per device
 * ordinal for the life of the process: calls after a cudaDeviceReset, or from a context other
 * than the device's primary context, are not supported (the kept address belongs to the old
 * context). With err_word = NULL a device-side fault is recorded only inside the scratch, where
 * no call can read it: pass an err_word to see it. */
k3moe_status k3moe_route_noalloc(const k3moe_dims* dims, const uint16_t* x, int32_t T,
                                 const uint16_t* w_router, const float* bias, int32_t* topk_idx,
                                 float* topk_w, uint32_t* err_word, void* stream);

/* Token-by-expert permutation: histogram over experts, exclusive scan, stable scatter. The
 * pages route each token to 16 of 896 experts ("kimi-k3-mlx", Architecture table) and run each
 * expert once over the rows routed to it; this call groups the (token, slot) pairs by expert so
 * that an expert's weights are read once per step. Rows of one expert keep token order, so the
 * result is deterministic and equals a two-pass counting sort.
 *   topk_idx [T][k] int32 in [0, E): each token's experts, distinct.
 *   expert_offsets [E+1] out: rows of expert e are [offsets[e], offsets[e+1]).
 *   row_token, row_slot [T*k] out: the (token, slot) behind sorted row r; rows of one
 *   expert are in ascending token order. slot_row [T*k] out: sorted row of pair (t, j). */
k3moe_status k3moe_permute(const k3moe_dims* dims, const int32_t* topk_idx, int32_t T,
                           int32_t* expert_offsets, int32_t* row_token, int32_t* row_slot,
                           int32_t* slot_row, void* ws, size_t ws_bytes, void* stream);

/* Dense bf16 projection out = bf16(W x) per token: the latent in (W_in [L][H]) and latent
 * out (W_out [H][L]) steps of Stable LatentMoE ("kimi-k3-mlx", LatentMoE: routed experts
 * compress the 7168-wide residual to 3584).
 *   W [N][K] bf16, x [T][K] bf16, out [T][N] bf16; N, K positive multiples of 64. */
k3moe_status k3moe_project(const uint16_t* W, const uint16_t* x, int32_t T, int32_t N,
                           int32_t K, uint16_t* out, void* ws, size_t ws_bytes, void* stream);

/* Routed expert FFN over the permuted rows ("kimi-k3-in-c", MXFP4 experts):
 *   for each sorted row r of expert e with token t = row_token[r]:
 *   o_rows[r] = D_e bf16(act(G_e z_t) * (U_e z_t))   (fp32 accumulation, fp32 GLU)
 *   z [T][L] bf16; expert_offsets [E+1], row_token [T*k] as from k3moe_permute;
 *   o_rows [T*k][L] fp32 out, in sorted-row order. */
k3moe_status k3moe_expert_ffn_mxfp4(const k3moe_dims* dims, const k3moe_weights* weights,
                                    const uint16_t* z, int32_t T, const int32_t* expert_offsets,
                                    const int32_t* row_token, float* o_rows, void* ws,
                                    size_t ws_bytes, void* stream);

/* Routing-weighted combine in latent space: c[t] = bf16(sum_{j<k} w[t][j] o_rows[slot_row[t*k+j]]),
 * summed in fp32 with j ascending ("kimi-k3-mlx", Architecture table and LatentMoE: the routed
 * experts' outputs are mixed by the router's renormalised weights in the 3584-wide latent space,
 * before the projection back to the residual). o_rows [T*k][L] fp32, slot_row [T*k],
 * topk_w [T][k], c [T][L] bf16 out. */
k3moe_status k3moe_combine(const k3moe_dims* dims, const float* o_rows, const int32_t* slot_row,
                           const float* topk_w, int32_t T, uint16_t* c, void* stream);

/* The whole layer: x [T][H] bf16 -> y [T][H] bf16, the routed experts plus, when
 * dims->n_shared > 0, the shared experts (y = bf16(W_out c + s), one rounding). topk_idx_out
 * [T][k] and topk_w_out [T][k] may be NULL; when given they receive the routing decisions.
 * Neither allocates nor synchronises: the call can be captured in a CUDA graph. */
k3moe_status k3moe_layer_forward(const k3moe_dims* dims, const k3moe_weights* weights,
                                 const uint16_t* x, int32_t T, uint16_t* y,
                                 int32_t* topk_idx_out, float* topk_w_out, void* ws,
                                 size_t ws_bytes, void* stream);

/* Prepared layer (optional, once per layer, outside the hot path). k3moe_layer_init checks dims
 * and weights as k3moe_layer_forward does and keeps a copy of both (the weight buffers must
 * outlive the handle). When latent and inter are multiples of 128 it also repacks the expert
 * scales gate_s, up_s and down_s into the image the expert kernels copy to tensor memory: for
 * every 128 weight rows and 128 codes of K, one 512-byte block whose byte 16 l + 4 w + q is the
 * scale of row 32 w + l, K-block 4 c + q; and gate_s with up_s once more, interleaved per 64
 * features (rows 0..63 of a block the gate rows, 64..127 the up rows of the same features) for
 * the many-token GLU tile. Those copies (twice the gate and up scale bytes plus the down scale
 * bytes) are device memory the handle owns; init allocates them, launches the repacking on
 * `stream` and synchronises the stream. On failure *layer is NULL and nothing is kept.
 * k3moe_layer_run is k3moe_layer_forward on the prepared layer, with the same arguments after
 * the handle and the same results bit for bit; the expert kernels then load each stage's weight
 * scales with one bulk copy next to the weight tile instead of gathering them row by row. It
 * neither allocates nor synchronises. k3moe_layer_free releases the handle and its
 * device memory (NULL is accepted; it synchronises the device while freeing). */
typedef struct k3moe_layer k3moe_layer;
k3moe_status k3moe_layer_init(const k3moe_dims* dims, const k3moe_weights* weights, k3moe_layer** layer,
                              void* stream);
k3moe_status k3moe_layer_run(const k3moe_layer* layer, const uint16_t* x, int32_t T, uint16_t* y,
                             int32_t* topk_idx_out, float* topk_w_out, void* ws, size_t ws_bytes,
                             void* stream);
/* k3moe_layer_run on host buffers: x_host [T][hidden] and y_host [T][hidden] (bf16 bits) are
 * page-locked host memory mapped into the device's address space (cudaMallocHost, cudaHostAlloc
 * or cudaHostRegister on a system with unified addressing); topk_idx_out / topk_w_out (optional)
 * and ws stay device memory. A kernel reads the tokens from host memory into the workspace
 * over the CPU-GPU link, the layer runs as k3moe_layer_run (same bits), and a kernel writes
 * y into y_host: no DMA copy call, and the three launches chain like the layer's own. y_host
 * holds the result once `stream` has completed. K3MOE_E_HOSTMEM if either buffer is not such
 * memory (checked on the host: nothing is launched), K3MOE_E_ALIGN if its device address is not
 * 16-byte aligned, K3MOE_E_SHAPE if T * hidden * 2 is not a multiple of 16. */
k3moe_status k3moe_layer_run_host(const k3moe_layer* layer, const uint16_t* x_host, int32_t T, uint16_t* y_host,
                                  int32_t* topk_idx_out, float* topk_w_out, void* ws, size_t ws_bytes,
                                  void* stream);
k3moe_status k3moe_layer_free(k3moe_layer* layer);

/* Synchronises `stream`, reads and clears the workspace error word. Returns K3MOE_OK,
 * K3MOE_E_TIMEOUT (a bounded wait ran out) or K3MOE_E_DEVICE (another device-side check),
 * or K3MOE_E_CUDA if the stream reported an error. */
k3moe_status k3moe_check(void* ws, void* stream);

/* After k3moe_layer_forward or k3moe_permute + k3moe_expert_ffn_mxfp4 on T tokens with this
 * workspace and dims: synchronises `stream` and reports how many distinct experts the step
 * selected (*distinct) and the expert bytes that step had to read, distinct x the bytes of one
 * expert (*expert_bytes; 17,547,264 per expert at K3 sizes). Either output may be NULL. Host
 * pointers; K3MOE_E_CUDA if the stream reported an error. */
k3moe_status k3moe_layer_stats(const k3moe_dims* dims, int32_t T, void* ws, size_t ws_bytes, void* stream,
                               int32_t* distinct, int64_t* expert_bytes);

/* REAP saliency accumulation ("kimi-k3-mlx" digest, REAP pruning section: expert j's saliency
 * S_j = (1/|C|) sum over calibration tokens x of g_j(x) * ||e_j(x)||_2). After
 * k3moe_layer_forward on T tokens with this workspace, adds w[t][j] * ||o_tj||_2 to
 * saliency[e] for every token t and slot j of that step, e = topk_idx[t][j], where o_tj is the
 * expert's fp32 output row in the latent space (before the combine) and w the renormalised
 * routing weight. Dividing the accumulated sums by the number of tokens gives S_j.
 *   topk_idx [T][k], topk_w [T][k]: the routing the layer call returned through topk_idx_out /
 *   topk_w_out, or NULL for the workspace's own copies (valid when that call passed NULL).
 *   saliency [E] fp64, device, accumulated into; fp64 atomic adds, so the order of the
 *   additions (and the last bits of the sums) varies between runs.
 * Reads the step's expert rows from the workspace: call it before the workspace is reused. */
k3moe_status k3moe_layer_saliency(const k3moe_dims* dims, int32_t T, const int32_t* topk_idx, const float* topk_w,
                                  void* ws, size_t ws_bytes, double* saliency, void* stream);

/* Human-readable name of a status code (static string). */
const char* k3moe_status_string(k3moe_status status);

/* Failure-detection self test (diagnostic; no counterpart on the pages): enqueues one kernel
 * whose single thread waits on a shared-memory barrier that nothing completes, with the same
 * bounded wait every kernel of the library uses (about 2 s of wall clock). The wait runs out,
 * the kernel records a timeout in the workspace error word and returns; the context stays
 * usable and the next k3moe_check reports K3MOE_E_TIMEOUT (and clears the word). `ws` is a
 * device workspace of at least 256 bytes. Returns K3MOE_E_CUDA if the launch fails. */
k3moe_status k3moe_selftest_timeout(void* ws, void* stream);

/* Scheduling self test (diagnostic; no counterpart on the pages): enqueues n_ctas CTAs, each
 * holding about 200 KB of shared memory (so no other large-shared-memory CTA fits beside it on
 * its SM) while one thread waits on the wall clock for `ms` milliseconds; then they exit. It
 * stands for other work that keeps SMs from the layer's kernels, e.g. on another stream.
 * 1 <= n_ctas <= 4096, 1 <= ms <= 10000 (K3MOE_E_SHAPE otherwise); K3MOE_E_CUDA if the launch
 * fails. */
k3moe_status k3moe_selftest_occupy(int32_t n_ctas, int32_t ms, void* stream);

/* Diagnostic per-kernel timing of k3moe_layer_forward (not needed for normal use; no
 * counterpart on the pages). mode = 1 starts recording: every kernel launch of later
 * layer_forward calls is bracketed by CUDA events on the caller's stream. mode = 0 stops,
 * synchronises those events and writes, for kernel ids 0 .. n-1, the summed milliseconds
 * (total_ms[n]) and launch counts (launches[n]); either array may be NULL. Returns
 * K3MOE_E_CUDA if an event call fails. Kernel names: k3moe_profile_name(id), NULL past the
 * last id. Not thread-safe; recording holds at most 65,536 launches. */
k3moe_status k3moe_profile(int32_t mode, int32_t n, float* total_ms, int32_t* launches);
const char* k3moe_profile_name(int32_t id);

#ifdef __cplusplus
}
#endif

#endif /* K3MOE_H */
