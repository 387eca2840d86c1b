/*
 * Reference oracle for one Stable-LatentMoE routed-expert layer with MXFP4 experts.
 *
 * TEST INFRASTRUCTURE ONLY. This is the plain, slow, obviously correct CPU statement of
 * what the CUDA library computes. Only the tests, the smoke check and the bench's CPU
 * baseline may load it; the library never calls it and shares no code with it.
 *
 * Sources (page title, then the section or table):
 *  - "kimi-k3-mlx" digest, "Architecture" table: 896 routed experts, top-16 per token,
 *    routed experts run in a 3584-wide latent space instead of the 7168-wide residual;
 *    the activation is SiTU-GLU (beta = 4, beta_lin = 25), evaluated in fp32.
 *  - same page, "Quantisation tiers": experts are MXFP4, low-nibble-first codes with
 *    e8m0 scales, reinterpreted without arithmetic.
 *  - "kimi-k3-in-c" (discuss.pytorch.kr), "MXFP4 experts": each weight is a 4-bit nibble
 *    that indexes a 16-entry table; 32 consecutive weights share one 8-bit exponent;
 *    0.53125 bytes per weight; 33,030,144 parameters and 17,547,264 bytes per expert.
 *  - "Kimi K3 hardware deep dive" (Tokios), "Quantisation-aware training": MXFP4 weights
 *    with MXFP8 activations.
 * Readings where the pages are silent (each listed in the design notes):
 *  - e2m1 and e4m3 values and the e8m0 rule follow the OCP Microscaling (MX) v1.0 spec.
 *  - Scales run along K (the input dimension); matrices are row-major [N][K].
 *  - act = SiLU-GLU: a = silu(gate) * up (SiTU-GLU has no formula on the pages).
 *  - Routing: softmax over all logits, top-k, renormalise over the k kept. Selection is
 *    on the logits (ties -> lowest index); indices are reported in ascending order.
 *  - One shared latent-in W_in [L][H] and latent-out W_out [H][L] per layer; the combine
 *    runs in latent space before W_out.
 *  - bf16 round-to-nearest-even at z, at the GLU output a, at the combine c and at y.
 *  - MXFP4 activations (actq = 2, the 4-bit activation mode that the fp4 tensor rate needs;
 *    the library does not run it yet): z and a go through an OCP MX FP4 round trip (e2m1
 *    elements, shared exponent floor(log2 amax) - 2, round-to-nearest-even, saturating at 6)
 *    where the MXFP8 mode applies its E4M3 round trip.
 *  - Shared experts ("kimi-k3-mlx", Architecture table and LatentMoE: n_shared always-on
 *    experts per token that work on the H-wide residual, not in the latent space; the
 *    weights outside the routed experts are bf16, Quantisation tiers): each is a bf16 GLU
 *    FFN with the routed experts' activation, s_j = D_j bf16(silu(G_j x) * (U_j x)); their
 *    width is not on the pages (a parameter). The shared outputs are added to W_out c before
 *    the one rounding of y: y = bf16(W_out c + sum_j s_j).
 * Arithmetic: every sum in double; decode is scalar, element by element.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
  int32_t hidden, latent, inter, n_experts, top_k;
  int32_t act;   /* 0 = SiLU-GLU */
  int32_t actq;  /* 0 = bf16 activations, 1 = MXFP8, 2 = MXFP4 (e2m1 + e8m0 per 32) */
  int32_t n_shared;      /* always-on shared experts (0 = none) */
  int32_t shared_inter;  /* intermediate width of each shared expert */
} k3o_dims;

/* Expert tensors are passed as tables of n_experts pointers (NULL for an expert that is
 * never selected), each pointing at that expert's row-major array. */
typedef struct {
  const uint16_t* w_router;   /* [E][H] bf16 */
  const float* router_bias;   /* [E] or NULL */
  const uint16_t* w_in;       /* [L][H] bf16 */
  const uint16_t* w_out;      /* [H][L] bf16 */
  const uint8_t* const* gate_q; /* per expert [I][L/2] */
  const uint8_t* const* gate_s; /* per expert [I][L/32] */
  const uint8_t* const* up_q;
  const uint8_t* const* up_s;
  const uint8_t* const* down_q; /* per expert [L][I/2] */
  const uint8_t* const* down_s; /* per expert [L][I/32] */
  /* shared experts, stacked: expert j owns rows [j*Is, (j+1)*Is) of gate/up and the same
   * columns of down (Is = shared_inter, S = n_shared * Is) */
  const uint16_t* w_sgate;    /* [S][H] bf16 */
  const uint16_t* w_sup;      /* [S][H] bf16 */
  const uint16_t* w_sdown;    /* [H][S] bf16 */
} k3o_weights;

/* ------------------------------------------------------------------ number formats */

/* bf16 -> double: bf16 is the top half of an IEEE binary32. */
double k3o_bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* double -> bf16, round to nearest, ties to even, in one step (no intermediate float).
 * bf16: 1 sign, 8 exponent (bias 127), 7 fraction bits; subnormals below 2^-126. */
uint16_t k3o_bf16_from_double(double x) {
  if (isnan(x)) return 0x7fc0;
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  double a = fabs(x);
  if (a == 0.0) return sign;
  if (isinf(a)) return sign | 0x7f80;
  int e;
  frexp(a, &e);                 /* a = f * 2^e, f in [0.5, 1) -> a in [2^(e-1), 2^e) */
  int exp2 = e - 1;             /* a in [2^exp2, 2^(exp2+1)) */
  if (exp2 < -126) exp2 = -126; /* subnormal range: fixed quantum 2^-133 */
  double quantum = ldexp(1.0, exp2 - 7);
  double m = a / quantum;       /* exact: scaling by a power of two */
  double r = nearbyint(m);      /* default rounding mode: nearest, ties to even */
  double v = r * quantum;
  if (v >= ldexp(1.0, 128)) return sign | 0x7f80; /* overflow to infinity */
  /* re-encode the exact value v */
  float vf = (float)v;          /* exact: v has <= 8 significant bits and is in range */
  uint32_t u;
  memcpy(&u, &vf, 4);
  return sign | (uint16_t)(u >> 16);
}

/* e2m1 (OCP MX v1.0, FP4): 1 sign bit (bit 3), 2 exponent bits (bias 1), 1 mantissa bit.
 * Exponent field 0 is subnormal: value = m * 2^(1-1) * 0.5. */
double k3o_e2m1(int code) {
  int s = (code >> 3) & 1, ex = (code >> 1) & 3, m = code & 1;
  /* 2^(ex-1) for ex in {1, 2, 3} is 1, 2 or 4: an exact small integer */
  double mag = (ex == 0) ? 0.5 * m : (1.0 + 0.5 * m) * (double)(1 << (ex - 1));
  return s ? -mag : mag;
}

/* e8m0 (OCP MX v1.0 shared scale): 2^(E-127); E = 255 is NaN. */
double k3o_e8m0(int e) {
  if (e == 255) return NAN;
  return ldexp(1.0, e - 127);
}

/* e4m3 (OCP MX v1.0, FP8 E4M3): bias 7, no infinities, S.1111.111 is NaN,
 * exponent field 0 is subnormal with quantum 2^-9. */
double k3o_e4m3(int code) {
  int s = (code >> 7) & 1, ex = (code >> 3) & 15, m = code & 7;
  double mag;
  if (ex == 15 && m == 7) return NAN;
  if (ex == 0) mag = ldexp((double)m, -9);
  else mag = ldexp(1.0 + m / 8.0, ex - 7);
  return s ? -mag : mag;
}

/* Round a real value to e4m3 with round-to-nearest-even, saturating to +-448 (the
 * conversion the OCP MX spec prescribes for FP8 elements). Returns the code. */
int k3o_e4m3_encode(double v) {
  if (isnan(v)) return 0x7f;
  int s = signbit(v) ? 1 : 0;
  double a = fabs(v);
  double q;
  if (a >= 448.0) {
    q = 448.0;
  } else if (a == 0.0) {
    q = 0.0;
  } else {
    int e;
    frexp(a, &e);
    int exp2 = e - 1;
    if (exp2 < -6) exp2 = -6;            /* subnormals share the quantum of 2^-6 * 2^-3 */
    double quantum = ldexp(1.0, exp2 - 3);
    q = nearbyint(a / quantum) * quantum;
    if (q > 448.0) q = 448.0;
  }
  /* find the code of q by search over the 127 non-negative finite codes */
  for (int c = 0; c < 127; ++c)
    if (k3o_e4m3(c) == q) return (s << 7) | c;
  return 0x7f; /* unreachable */
}

/* MXFP8 quantisation of one block of 32 values (OCP MX v1.0, section on conversion):
 * shared exponent X = floor(log2(amax)) - emax_elem, emax_elem = 8 for E4M3, clamped to
 * the e8m0 range [-127, 127]; elements are v / 2^X rounded to e4m3 (RNE, saturating).
 * An all-zero block gets X = -127 and zero elements. */
void k3o_mxfp8_block(const double* v, uint8_t* codes, uint8_t* scale_e8m0) {
  double amax = 0.0;
  for (int i = 0; i < 32; ++i)
    if (fabs(v[i]) > amax) amax = fabs(v[i]);
  int X;
  if (amax == 0.0 || !isfinite(amax)) {
    X = (amax == 0.0) ? -127 : 127;
  } else {
    int e;
    frexp(amax, &e);
    X = (e - 1) - 8;
    if (X < -127) X = -127;
    if (X > 127) X = 127;
  }
  *scale_e8m0 = (uint8_t)(X + 127);
  for (int i = 0; i < 32; ++i) codes[i] = (uint8_t)k3o_e4m3_encode(ldexp(v[i], -X));
}

/* Value after MXFP8 round trip, in place, for a vector whose length is a multiple of 32. */
void k3o_mxfp8_roundtrip(double* v, int n) {
  uint8_t codes[32], sc;
  for (int b = 0; b < n; b += 32) {
    k3o_mxfp8_block(v + b, codes, &sc);
    for (int i = 0; i < 32; ++i) v[b + i] = k3o_e4m3(codes[i]) * k3o_e8m0(sc);
  }
}

/* Round a real value to e2m1 with round-to-nearest-even, saturating to +-6 (the element
 * conversion of the OCP MX spec for FP4). Returns the 4-bit code. */
int k3o_e2m1_encode(double v) {
  const int s = signbit(v) ? 8 : 0;
  const double a = fabs(v);
  if (isnan(v)) return s | 7; /* no NaN in e2m1: saturate */
  /* the 8 magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6 at codes 0..7; pick the nearest, ties to the
   * even code */
  int best = 0;
  double bd = INFINITY;
  for (int c = 0; c < 8; ++c) {
    const double d = fabs(a - k3o_e2m1(c));
    if (d < bd || (d == bd && (c & 1) == 0)) {
      bd = d;
      best = c;
    }
  }
  return s | best;
}

/* MXFP4 quantisation of one block of 32 values (OCP MX v1.0 conversion, FP4 E2M1 elements):
 * shared exponent X = floor(log2(amax)) - emax_elem, emax_elem = 2 for E2M1, clamped to the
 * e8m0 range [-127, 127]; elements are v / 2^X rounded to e2m1 (RNE, saturating at 6). An
 * all-zero block gets X = -127 and zero elements. */
void k3o_mxfp4_block(const double* v, uint8_t* codes, uint8_t* scale_e8m0) {
  double amax = 0.0;
  for (int i = 0; i < 32; ++i)
    if (fabs(v[i]) > amax) amax = fabs(v[i]);
  int X;
  if (amax == 0.0 || !isfinite(amax)) {
    X = (amax == 0.0) ? -127 : 127;
  } else {
    int e;
    frexp(amax, &e);
    X = (e - 1) - 2;
    if (X < -127) X = -127;
    if (X > 127) X = 127;
  }
  *scale_e8m0 = (uint8_t)(X + 127);
  for (int i = 0; i < 32; ++i) codes[i] = (uint8_t)k3o_e2m1_encode(ldexp(v[i], -X));
}

/* Value after MXFP4 round trip, in place, for a vector whose length is a multiple of 32. */
void k3o_mxfp4_roundtrip(double* v, int n) {
  uint8_t codes[32], sc;
  for (int b = 0; b < n; b += 32) {
    k3o_mxfp4_block(v + b, codes, &sc);
    for (int i = 0; i < 32; ++i) v[b + i] = k3o_e2m1(codes[i]) * k3o_e8m0(sc);
  }
}

/* Weight j of one MXFP4 row: code = nibble j (low nibble first), scale = byte j/32. */
double k3o_mx_weight(const uint8_t* q_row, const uint8_t* s_row, int j) {
  int byte = q_row[j / 2];
  int code = (j % 2 == 0) ? (byte & 0xF) : ((byte >> 4) & 0xF);
  return k3o_e2m1(code) * k3o_e8m0(s_row[j / 32]);
}

/* One MXFP4 row of K weights to doubles: block b of 32 consecutive weights shares the scale
 * s_row[b]; weight j is the nibble j (low nibble first) times that scale. */
void k3o_dequant_row(const uint8_t* q_row, const uint8_t* s_row, int K, double* out) {
  double table[16]; /* the 16-entry value table the nibbles index */
  for (int c = 0; c < 16; ++c) table[c] = k3o_e2m1(c);
  for (int b = 0; b < K / 32; ++b) {
    const double scale = k3o_e8m0(s_row[b]);
    for (int i = 0; i < 32; ++i) {
      const int j = 32 * b + i;
      const int byte = q_row[j / 2];
      const int code = (j % 2 == 0) ? (byte & 0xF) : ((byte >> 4) & 0xF);
      out[j] = table[code] * scale;
    }
  }
}

/* Whole MXFP4 matrix [N][K] to doubles (row-major), row by row. */
void k3o_dequant(const uint8_t* q, const uint8_t* s, int N, int K, double* out) {
  for (int n = 0; n < N; ++n)
    k3o_dequant_row(q + (size_t)n * (K / 2), s + (size_t)n * (K / 32), K, out + (size_t)n * K);
}

/* ------------------------------------------------------------------ sizes (pins) */
int64_t k3o_expert_params(const k3o_dims* d) { return 3LL * d->latent * d->inter; }
/* Bytes of one expert: half a byte per code plus one scale byte per 32 codes. */
int64_t k3o_expert_bytes(const k3o_dims* d) {
  int64_t p = k3o_expert_params(d);
  return p / 2 + p / 32;
}

/* ------------------------------------------------------------------ layer steps */

/* Router logits l[t][e] = sum_h x[t][h] * W_r[e][h] + b[e], in double. */
void k3o_router_logits(const k3o_dims* d, const uint16_t* x, int T, const uint16_t* w_router,
                       const float* bias, double* logits) {
  const int H = d->hidden, E = d->n_experts;
  for (int t = 0; t < T; ++t)
    for (int e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int h = 0; h < H; ++h)
        acc += k3o_bf16_to_double(x[(size_t)t * H + h]) *
               k3o_bf16_to_double(w_router[(size_t)e * H + h]);
      if (bias) acc += (double)bias[e];
      logits[(size_t)t * E + e] = acc;
    }
}

/* Selection of the k largest logits of one token: sort the pairs (-l, e)
 * lexicographically (ties -> lower index first, NaN ordered last) and keep the first k;
 * the kept indices are returned in ascending order. */
typedef struct { double l; int e; } k3o_pair;
static int k3o_pair_cmp(const void* a, const void* b) {
  const k3o_pair* p = (const k3o_pair*)a;
  const k3o_pair* q = (const k3o_pair*)b;
  int pn = isnan(p->l), qn = isnan(q->l);
  if (pn != qn) return pn - qn;
  if (!pn && p->l != q->l) return (p->l > q->l) ? -1 : 1;
  return p->e - q->e;
}
static int k3o_int_cmp(const void* a, const void* b) {
  return *(const int32_t*)a - *(const int32_t*)b;
}
void k3o_select_topk(const double* logits, int T, int E, int k, int32_t* idx) {
  k3o_pair* p = (k3o_pair*)malloc(sizeof(k3o_pair) * (size_t)E);
  for (int t = 0; t < T; ++t) {
    for (int e = 0; e < E; ++e) { p[e].l = logits[(size_t)t * E + e]; p[e].e = e; }
    qsort(p, (size_t)E, sizeof(k3o_pair), k3o_pair_cmp);
    for (int j = 0; j < k; ++j) idx[(size_t)t * k + j] = p[j].e;
    qsort(idx + (size_t)t * k, (size_t)k, sizeof(int32_t), k3o_int_cmp);
  }
  free(p);
}

/* Routing weights: softmax over all E logits, then renormalised over the kept k. */
void k3o_route_weights(const double* logits, const int32_t* idx, int T, int E, int k, double* w) {
  for (int t = 0; t < T; ++t) {
    const double* l = logits + (size_t)t * E;
    double mx = -INFINITY;
    for (int e = 0; e < E; ++e) if (l[e] > mx) mx = l[e];
    double z = 0.0;
    for (int e = 0; e < E; ++e) z += exp(l[e] - mx);
    double kept = 0.0;
    for (int j = 0; j < k; ++j) kept += exp(l[idx[(size_t)t * k + j]] - mx) / z;
    for (int j = 0; j < k; ++j)
      w[(size_t)t * k + j] = (exp(l[idx[(size_t)t * k + j]] - mx) / z) / kept;
  }
}

/* Token-by-expert permutation as a two-pass counting sort: count rows per expert,
 * exclusive prefix sum, then append (t, slot) pairs in token order, slot order.
 * offsets[E+1]; row_token/row_slot[T*k] give the pair behind sorted row r;
 * slot_row[t*k + j] gives the sorted row of pair (t, j). */
void k3o_permute(const int32_t* idx, int T, int E, int k, int32_t* offsets, int32_t* row_token,
                 int32_t* row_slot, int32_t* slot_row) {
  int32_t* fill = (int32_t*)calloc((size_t)E, sizeof(int32_t));
  for (int e = 0; e <= E; ++e) offsets[e] = 0;
  for (int i = 0; i < T * k; ++i) offsets[idx[i] + 1] += 1;
  for (int e = 0; e < E; ++e) offsets[e + 1] += offsets[e];
  for (int t = 0; t < T; ++t)
    for (int j = 0; j < k; ++j) {
      int e = idx[(size_t)t * k + j];
      int r = offsets[e] + fill[e]++;
      row_token[r] = t;
      row_slot[r] = j;
      slot_row[(size_t)t * k + j] = r;
    }
  free(fill);
}

/* Dense bf16 projection out[t][n] = sum_k W[n][k] * x[t][k] (double); optional bf16 copy. */
void k3o_dense_proj(const uint16_t* W, const uint16_t* x, int T, int N, int K, double* out,
                    uint16_t* out_bf16) {
  for (int t = 0; t < T; ++t)
    for (int n = 0; n < N; ++n) {
      double acc = 0.0;
      for (int k = 0; k < K; ++k)
        acc += k3o_bf16_to_double(W[(size_t)n * K + k]) * k3o_bf16_to_double(x[(size_t)t * K + k]);
      if (out) out[(size_t)t * N + n] = acc;
      if (out_bf16) out_bf16[(size_t)t * N + n] = k3o_bf16_from_double(acc);
    }
}

static double k3o_silu(double g) { return g / (1.0 + exp(-g)); }

/* One routed row through expert e: z (bf16, [L]) -> o (double, [L]).
 *   g = G_e z, u = U_e z             (MXFP8 mode: z first goes through MXFP8)
 *   a = bf16(silu(g) * u)            (MXFP8 mode: a then goes through MXFP8)
 *   o = D_e a
 * `a_out` (optional, [I]) receives a as bf16. Returns 0, or -1 for an unsupported act. */
int k3o_expert_row(const k3o_dims* d, const k3o_weights* w, int e, const uint16_t* z,
                   double* o, uint16_t* a_out) {
  const int L = d->latent, I = d->inter;
  if (d->act != 0) return -1;
  double* zin = (double*)malloc(sizeof(double) * (size_t)L);
  double* a = (double*)malloc(sizeof(double) * (size_t)I);
  double* wg = (double*)malloc(sizeof(double) * (size_t)(L > I ? L : I));
  double* wu = (double*)malloc(sizeof(double) * (size_t)L);
  for (int k = 0; k < L; ++k) zin[k] = k3o_bf16_to_double(z[k]);
  if (d->actq == 1) k3o_mxfp8_roundtrip(zin, L);
  if (d->actq == 2) k3o_mxfp4_roundtrip(zin, L);
  const uint8_t *gq = w->gate_q[e], *gs = w->gate_s[e], *uq = w->up_q[e], *us = w->up_s[e];
  for (int n = 0; n < I; ++n) {
    double g = 0.0, u = 0.0;
    k3o_dequant_row(gq + (size_t)n * (L / 2), gs + (size_t)n * (L / 32), L, wg);
    k3o_dequant_row(uq + (size_t)n * (L / 2), us + (size_t)n * (L / 32), L, wu);
    for (int k = 0; k < L; ++k) {
      g += wg[k] * zin[k];
      u += wu[k] * zin[k];
    }
    uint16_t ab = k3o_bf16_from_double(k3o_silu(g) * u);
    if (a_out) a_out[n] = ab;
    a[n] = k3o_bf16_to_double(ab);
  }
  if (d->actq == 1) k3o_mxfp8_roundtrip(a, I);
  if (d->actq == 2) k3o_mxfp4_roundtrip(a, I);
  const uint8_t *dq = w->down_q[e], *ds = w->down_s[e];
  for (int n = 0; n < L; ++n) {
    double acc = 0.0;
    k3o_dequant_row(dq + (size_t)n * (I / 2), ds + (size_t)n * (I / 32), I, wg);
    for (int k = 0; k < I; ++k) acc += wg[k] * a[k];
    o[n] = acc;
  }
  free(zin);
  free(a);
  free(wg);
  free(wu);
  return 0;
}

/* The shared experts on one token x (bf16, [H]): s = sum_j D_j bf16(silu(G_j x) * (U_j x))
 * (double, [H]); `a_out` (optional, [S]) receives the stacked GLU outputs as bf16. Each expert
 * is summed on its own, in expert order. Returns 0, or -1 for an unsupported act. */
int k3o_shared_ffn(const k3o_dims* d, const k3o_weights* w, const uint16_t* x, double* s,
                   uint16_t* a_out) {
  const int H = d->hidden, Is = d->shared_inter;
  if (d->act != 0) return -1;
  double* a = (double*)malloc(sizeof(double) * (size_t)(Is > 0 ? Is : 1));
  for (int h = 0; h < H; ++h) s[h] = 0.0;
  for (int j = 0; j < d->n_shared; ++j) {
    for (int i = 0; i < Is; ++i) {
      const size_t r = (size_t)j * Is + i;
      double g = 0.0, u = 0.0;
      for (int k = 0; k < H; ++k) {
        const double xk = k3o_bf16_to_double(x[k]);
        g += k3o_bf16_to_double(w->w_sgate[r * H + k]) * xk;
        u += k3o_bf16_to_double(w->w_sup[r * H + k]) * xk;
      }
      const uint16_t ab = k3o_bf16_from_double(k3o_silu(g) * u);
      if (a_out) a_out[r] = ab;
      a[i] = k3o_bf16_to_double(ab);
    }
    const size_t S = (size_t)d->n_shared * Is;
    for (int h = 0; h < H; ++h) {
      double acc = 0.0;
      for (int i = 0; i < Is; ++i) acc += k3o_bf16_to_double(w->w_sdown[(size_t)h * S + (size_t)j * Is + i]) * a[i];
      s[h] += acc;
    }
  }
  free(a);
  return 0;
}

/* Routing-weighted combine of one token in latent space: c = bf16(sum_j w_j * o_j),
 * j ascending. */
void k3o_combine_token(int L, int k, const double* const* o_rows, const double* w, uint16_t* c,
                       double* c_exact) {
  for (int n = 0; n < L; ++n) {
    double acc = 0.0;
    for (int j = 0; j < k; ++j) acc += w[j] * o_rows[j][n];
    if (c_exact) c_exact[n] = acc;
    c[n] = k3o_bf16_from_double(acc);
  }
}

/* Whole layer for T tokens, tokens independent (OpenMP over tokens when nthreads > 1):
 *   logits -> top-k (on the double logits) -> weights -> z = bf16(W_in x)
 *   -> per slot: expert row -> combine c = bf16(sum w o) -> y = bf16(W_out c + s), with s the
 *   shared experts' output on x (0 when n_shared = 0).
 * Outputs (any may be NULL except y): idx [T][k], wts [T][k], logits [T][E],
 * z [T][L], c [T][L], y [T][H]. Returns 0, or -1 for an unsupported mode or a selected
 * expert whose tensors were not supplied. */
int k3o_layer_forward(const k3o_dims* d, const k3o_weights* w, const uint16_t* x, int T,
                      uint16_t* y, int32_t* idx_out, double* w_out, double* logits_out,
                      uint16_t* z_out, uint16_t* c_out, int nthreads) {
  const int H = d->hidden, L = d->latent, E = d->n_experts, k = d->top_k;
  if (d->act != 0 || d->actq < 0 || d->actq > 2) return -1;
  if (d->n_shared < 0 || (d->n_shared > 0 && (d->shared_inter <= 0 || !w->w_sgate || !w->w_sup || !w->w_sdown)))
    return -1;
  int bad = 0;
#ifdef _OPENMP
  if (nthreads < 1) nthreads = 1;
#pragma omp parallel for num_threads(nthreads) schedule(dynamic, 1) reduction(| : bad)
#endif
  for (int t = 0; t < T; ++t) {
    const uint16_t* xt = x + (size_t)t * H;
    double* lg = (double*)malloc(sizeof(double) * (size_t)E);
    int32_t* id = (int32_t*)malloc(sizeof(int32_t) * (size_t)k);
    double* wt = (double*)malloc(sizeof(double) * (size_t)k);
    uint16_t* z = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)L);
    uint16_t* c = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)L);
    double* o = (double*)malloc(sizeof(double) * (size_t)k * L);
    const double** orow = (const double**)malloc(sizeof(double*) * (size_t)k);
    k3o_router_logits(d, xt, 1, w->w_router, w->router_bias, lg);
    k3o_select_topk(lg, 1, E, k, id);
    k3o_route_weights(lg, id, 1, E, k, wt);
    k3o_dense_proj(w->w_in, xt, 1, L, H, NULL, z);
    for (int j = 0; j < k; ++j) {
      int e = id[j];
      if (!w->gate_q[e] || !w->gate_s[e] || !w->up_q[e] || !w->up_s[e] || !w->down_q[e] ||
          !w->down_s[e]) {
        bad = 1;
        memset(o + (size_t)j * L, 0, sizeof(double) * (size_t)L);
      } else {
        k3o_expert_row(d, w, e, z, o + (size_t)j * L, NULL);
      }
      orow[j] = o + (size_t)j * L;
    }
    k3o_combine_token(L, k, orow, wt, c, NULL);
    double* yo = (double*)malloc(sizeof(double) * (size_t)H);
    k3o_dense_proj(w->w_out, c, 1, H, L, yo, NULL);
    if (d->n_shared > 0) {
      double* sh = (double*)malloc(sizeof(double) * (size_t)H);
      k3o_shared_ffn(d, w, xt, sh, NULL);
      for (int h = 0; h < H; ++h) yo[h] += sh[h];
      free(sh);
    }
    for (int h = 0; h < H; ++h) y[(size_t)t * H + h] = k3o_bf16_from_double(yo[h]);
    free(yo);
    if (idx_out) memcpy(idx_out + (size_t)t * k, id, sizeof(int32_t) * (size_t)k);
    if (w_out) memcpy(w_out + (size_t)t * k, wt, sizeof(double) * (size_t)k);
    if (logits_out) memcpy(logits_out + (size_t)t * E, lg, sizeof(double) * (size_t)E);
    if (z_out) memcpy(z_out + (size_t)t * L, z, sizeof(uint16_t) * (size_t)L);
    if (c_out) memcpy(c_out + (size_t)t * L, c, sizeof(uint16_t) * (size_t)L);
    free(lg); free(id); free(wt); free(z); free(c); free(o); free(orow);
  }
  return bad ? -1 : 0;
}

/* REAP saliency ("kimi-k3-mlx" digest, REAP pruning section): S_j = (1/|C|) sum over the
 * calibration tokens x of g_j(x) * ||e_j(x)||_2, the router's weight for expert j times the
 * norm of that expert's output, averaged over the |C| tokens (g_j(x) = 0 where x does not
 * select j). Reading taken: g_j is the renormalised routing weight the combine uses, e_j(x) the
 * expert's output row in the latent space (o before the combine). This adds the sums of one
 * step to S[E]: for each token t and slot j, S[idx[t][j]] += w[t][j] * sqrt(sum_n o[t][j][n]^2);
 * the caller divides by the number of calibration tokens. o is [T][k][L] in slot order. */
void k3o_saliency_accumulate(const k3o_dims* d, int T, const int32_t* idx, const double* w, const double* o,
                             double* S) {
  const int k = d->top_k, L = d->latent;
  for (int t = 0; t < T; ++t)
    for (int j = 0; j < k; ++j) {
      const double* row = o + ((size_t)t * k + j) * (size_t)L;
      double ss = 0.0;
      for (int n = 0; n < L; ++n) ss += row[n] * row[n];
      S[idx[(size_t)t * k + j]] += w[(size_t)t * k + j] * sqrt(ss);
    }
}

int k3o_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
