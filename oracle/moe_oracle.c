/*
 * CPU oracle for the batched grouped-masked block-FP8 MoE expert forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check of the package
 * entry file and the CPU-baseline / reference legs of the benchmark may load
 * this library.  The product path (the CUDA library and its Python binding)
 * never calls it and shares no code, header or table with it.
 *
 * Everything here is the plain definition, written step by step, in the
 * order the pages state it:
 *
 *   vllm.model_executor.layers.fused_moe.prepare_megamoe
 *     _quantize_fp8_groups  -> S1 (e4m3), S2 (group scale), S3 (quantise)
 *     _pack_bytes           -> S4 (four UE8M0 exponents per int32)
 *     _store_topk, _eplb_kernel_args, prepare_megamoe_inputs
 *                           -> S5 (top-k repack, padding, EPLB replica map)
 *   vllm.model_executor.layers.fused_moe.experts.fused_humming_moe
 *     BatchedHummingGroupedExperts.apply, HummingExpertsBase.get_buffer_metas,
 *     HummingExpertsBase.process_input
 *                           -> S6 (batched layout), S7 (w13 GEMM, SiLU-and-mul,
 *                              requant, w2 GEMM)
 *     HummingIndexedExperts.apply (moe_fused_mul_sum), TopKWeightAndReduceDelegate
 *                           -> S8 (top-k weighted reduce)
 *
 * Precision.  The group-scale arithmetic of _quantize_fp8_groups is fp32 on
 * the page (the scale is bit-cast to a 32-bit unsigned integer), so S2/S3
 * run in fp32.  Every dot product and the SiLU are evaluated in fp64 (the
 * pages do not fix them); the buffers the pages declare as bf16
 * (gate_up_output, down_output, output) are rounded once, to nearest-even,
 * from the fp64 value.  No blocking, fusion or reordering is applied.
 *
 * Build: plain C11, no -ffast-math, -ffp-contract=off, optional OpenMP.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_ABI_VERSION 1

int orc_abi_version(void) { return ORC_ABI_VERSION; }

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* bit helpers                                                              */
/* ------------------------------------------------------------------------ */
static float f32_from_bits(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t bits_from_f32(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

/* bf16 is the upper half of an fp32 bit pattern. */
static float bf16_to_f32(uint16_t b) { return f32_from_bits((uint32_t)b << 16); }

/* Round an fp64 value to bf16 (8 significant bits, 8 exponent bits), ties to
 * even, in one rounding step.  Overflow gives +-inf, NaN gives a quiet NaN. */
uint16_t orc_bf16_from_f64(double v) {
  if (isnan(v)) return 0x7FC0;
  uint16_t sign = signbit(v) ? 0x8000 : 0;
  double a = fabs(v);
  if (a == 0.0) return sign;
  int ex;
  frexp(a, &ex);                  /* a = m * 2^ex, m in [0.5, 1) */
  int q = ex - 8;                 /* quantum exponent for 8 significant bits */
  if (q < -133) q = -133;         /* bf16 subnormal quantum is 2^-133 */
  double r = nearbyint(ldexp(a, -q)); /* default rounding mode: ties to even */
  double res = ldexp(r, q);
  if (res > 3.38953138925153547590470800371487866880e+38) return sign | 0x7F80; /* inf */
  uint32_t fb = bits_from_f32((float)res);   /* exact: res has <= 8 bits */
  return (uint16_t)(sign | (fb >> 16));
}

/* ------------------------------------------------------------------------ */
/* S1: FP8 E4M3 (OCP "E4M3": bias 7, 3 mantissa bits, no infinities,        */
/* S.1111.111 is NaN, largest finite 448, subnormals m * 2^-9).             */
/* The page casts with `.to(tl.float8e4nv)`; rounding is to nearest, ties   */
/* to even, and magnitudes beyond 448 saturate to 448.                      */
/* ------------------------------------------------------------------------ */
float orc_e4m3_decode(uint8_t code) {
  int s = code >> 7, e = (code >> 3) & 0xF, m = code & 7;
  if (e == 15 && m == 7) return NAN;
  double mag = (e == 0) ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
  return (float)(s ? -mag : mag);
}

/* Encode |v| by searching the sorted table of the 127 non-negative finite
 * codes 0x00..0x7E (their values increase with the code). */
uint8_t orc_e4m3_encode(float v) {
  if (isnan(v)) return 0x7F;
  uint8_t sign = signbit(v) ? 0x80 : 0;
  double a = fabs((double)v);
  if (a >= 448.0) return sign | 0x7E;            /* satfinite */
  int lo = 0, hi = 0x7E;                         /* largest c with val(c) <= a */
  while (lo < hi) {
    int mid = (lo + hi + 1) / 2;
    if ((double)orc_e4m3_decode((uint8_t)mid) <= a) lo = mid; else hi = mid - 1;
  }
  int c = lo;
  double below = orc_e4m3_decode((uint8_t)c);
  if (below == a) return sign | (uint8_t)c;
  double above = orc_e4m3_decode((uint8_t)(c + 1));
  double d_lo = a - below, d_hi = above - a;
  int pick;
  if (d_lo < d_hi) pick = c;
  else if (d_hi < d_lo) pick = c + 1;
  else pick = (c % 2 == 0) ? c : c + 1;          /* tie: even code = even mantissa */
  return sign | (uint8_t)pick;
}

/* ------------------------------------------------------------------------ */
/* S2: group scale (fp32).  amax floored at 1e-4, scale = amax / 448.       */
/* UE8M0: exponent field of the scale, plus one when the mantissa is not    */
/* zero (round the power of two up), clamped to [1, 254]; the quantisation  */
/* scale is that power of two.  FP32 mode keeps the scale itself.           */
/* `code` returns the exponent byte (UE8M0) or the fp32 bit pattern.        */
/* ------------------------------------------------------------------------ */
void orc_group_scale(float amax, int ue8m0, uint32_t* code, float* qs) {
  float a = fmaxf(amax, 1.0e-4f);
  float s = a / 448.0f;
  if (ue8m0) {
    uint32_t b = bits_from_f32(s);
    uint32_t e = ((b >> 23) & 0xFFu) + ((b & 0x7FFFFFu) != 0u ? 1u : 0u);
    if (e < 1u) e = 1u;
    if (e > 254u) e = 254u;
    *code = e;
    *qs = f32_from_bits(e << 23);
  } else {
    *code = bits_from_f32(s);
    *qs = s;
  }
}

/* S2 + S3 on one group of `n` fp32 values: q_i = e4m3(v_i * (1 / qs)). */
static void quantize_group_f32(const float* v, int n, int ue8m0, uint8_t* q,
                               uint32_t* code, float* qs_out) {
  float amax = 0.0f;
  for (int i = 0; i < n; ++i) amax = fmaxf(amax, fabsf(v[i]));
  float qs;
  orc_group_scale(amax, ue8m0, code, &qs);
  float inv = 1.0f / qs;
  for (int i = 0; i < n; ++i) q[i] = orc_e4m3_encode(v[i] * inv);
  if (qs_out) *qs_out = qs;
}

/* ------------------------------------------------------------------------ */
/* S1-S5: MegaMoE input staging in token order (prepare_megamoe_inputs).    */
/* hidden   : bf16 bit patterns, row-major [T, K]                            */
/* sf_mode  : 1 = UE8M0 packed 4 per int32 into x_sf[T, ceil(G/4)]           */
/*            2 = fp32 scales into x_sf[T, G]                                */
/* ids      : int32 or int64 [T, top_k]; weights fp32 [T, top_k]             */
/* EPLB     : l2p [num_logical, map_stride] int32, replica_count, load       */
/*            (all may be NULL: inert).                                      */
/* Returns 0, or 2 for a shape error (K not a multiple of 128).             */
/* ------------------------------------------------------------------------ */
int orc_prepare_inputs(int64_t T, int64_t K, int64_t top_k, const uint16_t* hidden,
                       const void* topk_ids, int ids_is_int64, const float* topk_weights,
                       const uint8_t* is_padding, int sf_mode, uint8_t* x, void* x_sf,
                       int64_t* ids_out, float* w_out, const int32_t* l2p,
                       int64_t num_logical, int64_t map_stride,
                       const int32_t* replica_count, int32_t* expert_load,
                       int64_t num_physical, int record_enabled, int64_t num_unpadded) {
  if (T == 0) return 0;
  if (K % 128 != 0) return 2;
  const int64_t G = K / 128;
  const int64_t W = (G + 3) / 4;
  (void)num_logical;
  (void)num_physical;

  /* S1-S4: quantise each 1x128 group of each token. */
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t) {
    float v[128];
    uint8_t q[128];
    if (sf_mode == 1)
      for (int64_t w = 0; w < W; ++w) ((int32_t*)x_sf)[t * W + w] = 0;
    for (int64_t g = 0; g < G; ++g) {
      for (int i = 0; i < 128; ++i) v[i] = bf16_to_f32(hidden[t * K + g * 128 + i]);
      uint32_t code;
      quantize_group_f32(v, 128, sf_mode == 1, q, &code, NULL);
      memcpy(x + t * K + g * 128, q, 128);
      if (sf_mode == 1) {
        /* S4: exponent of group g is byte g%4 of word g/4 (little-endian). */
        uint32_t* words = (uint32_t*)x_sf;
        words[t * W + g / 4] |= (code & 0xFFu) << (8 * (g % 4));
      } else {
        ((float*)x_sf)[t * G + g] = f32_from_bits(code);
      }
    }
  }

  /* S5: top-k repack.  Padding tokens are unrouted: id -1, weight 0. */
  for (int64_t t = 0; t < T; ++t) {
    int pad = is_padding ? (is_padding[t] != 0) : 0;
    for (int64_t j = 0; j < top_k; ++j) {
      int64_t id = ids_is_int64 ? ((const int64_t*)topk_ids)[t * top_k + j]
                                : (int64_t)((const int32_t*)topk_ids)[t * top_k + j];
      if (pad) id = -1;
      if (l2p && id >= 0) {
        /* Replica chosen per token: t mod replica_count[logical id]. */
        int64_t r = t % replica_count[id];
        id = l2p[id * map_stride + r];
        if (expert_load && record_enabled && t < num_unpadded) expert_load[id] += 1;
      }
      ids_out[t * top_k + j] = id;
      w_out[t * top_k + j] = pad ? 0.0f : topk_weights[t * top_k + j];
    }
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* S4b: shared-expert scale pages (prepare_megamoe_inputs with shared_x_sf  */
/* and shared_block_m; _shared_sf_row).  Token t sits in page block          */
/* t / B (B = shared_block_m), whose rows are padded to a multiple of 128.   */
/* Inside the block, position m = t % B is split into its 128-row page       */
/* (m / 128) and, within that page, into quarter q = (m % 128) / 32 and      */
/* offset i = m % 32; the page stores offset-major: row 4*i + q.  The        */
/* exponent byte of group g lands in column g.                               */
int64_t orc_shared_sf_row(int64_t t, int64_t block_m) {
  const int64_t padded = ((block_m + 127) / 128) * 128;
  const int64_t block = t / block_m;
  const int64_t m = t % block_m;
  const int64_t page = m / 128;
  const int64_t quarter = (m % 128) / 32;
  const int64_t offset = m % 32;
  return block * padded + page * 128 + 4 * offset + quarter;
}

/* x_sf_words: [T, ceil(G/4)] packed exponents (S4) of the token-order      */
/* staging; out: uint8 with strides (s0, s1); untouched outside the rows of  */
/* the T tokens.                                                            */
void orc_shared_sf(int64_t T, int64_t G, const int32_t* x_sf_words, int64_t block_m,
                   uint8_t* out, int64_t s0, int64_t s1) {
  const int64_t W = (G + 3) / 4;
  for (int64_t t = 0; t < T; ++t) {
    const int64_t row = orc_shared_sf_row(t, block_m);
    for (int64_t g = 0; g < G; ++g) {
      const uint32_t word = (uint32_t)x_sf_words[t * W + g / 4];
      out[row * s0 + g * s1] = (uint8_t)((word >> (8 * (g % 4))) & 0xFFu);
    }
  }
}

/* ------------------------------------------------------------------------ */
/* N1: FP4 E2M1 (OCP MX "E2M1": 1 sign, 2 exponent (bias 1), 1 mantissa    */
/* bit; no infinities or NaN).  Magnitudes of codes 0..7:                    */
/*   0, 0.5 (subnormal), 1, 1.5, 2, 3, 4, 6.                                 */
float orc_e2m1_decode(uint8_t code) {
  const int sign = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
  const double mag = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return (float)(sign ? -mag : mag);
}

/* Round to nearest, ties to the even code, saturate finite overflow to 6. */
uint8_t orc_e2m1_encode(float v) {
  const uint8_t sign = signbit(v) ? 0x8 : 0;
  const double a = fabs((double)v);
  if (a >= 6.0) return sign | 0x7;
  int c = 0;                                     /* largest code with val <= a */
  while (c < 7 && (double)orc_e2m1_decode((uint8_t)(c + 1)) <= a) ++c;
  const double below = orc_e2m1_decode((uint8_t)c);
  if (below == a) return sign | (uint8_t)c;
  const double above = orc_e2m1_decode((uint8_t)(c + 1));
  const double d_lo = a - below, d_hi = above - a;
  int pick;
  if (d_lo < d_hi) pick = c;
  else if (d_hi < d_lo) pick = c + 1;
  else pick = (c % 2 == 0) ? c : c + 1;
  return sign | (uint8_t)pick;
}

/* N2: NVFP4 staging of one token row (prepare_megamoe_nvfp4_inputs,         */
/* kNvfp4DynamicToken): the row is scaled by its own fp32 x_scale = amax /   */
/* 2688 (2688 = 448 * 6, the largest E4M3 scale times the largest E2M1      */
/* value) and quantised to E2M1 with one E4M3 scale per 16 values.  Reading */
/* (the kernel body is not on the pages), in fp32 with IEEE roundings:       */
/*   xs = amax / 2688;  inv = 1 / xs;  v_i = x_i * inv   (|v| <= 2688)       */
/*   per 16 values: s = e4m3(max|v_i| / 6);  q_i = e2m1(v_i * (1 / dec(s)))  */
/* amax == 0 gives xs = 0 and zero codes; a block whose scale rounds to 0    */
/* gives zero codes.  Codes are packed two per byte (value 2i in the low    */
/* nibble), scales four per int32 (block b in byte b % 4 of word b / 4).     */
void orc_nvfp4_row(int64_t K, const uint16_t* hidden_row, uint8_t* x_row, int32_t* sf_row,
                   float* x_scale) {
  if (K <= 0) return;
  const int64_t nb = K / 16;
  float amax = 0.0f;
  for (int64_t i = 0; i < K; ++i) {
    const float a = fabsf(bf16_to_f32(hidden_row[i]));
    if (a > amax) amax = a;
  }
  const float xs = amax / 2688.0f;
  *x_scale = xs;
  memset(x_row, 0, (size_t)K / 2);
  memset(sf_row, 0, ((size_t)nb + 3) / 4 * 4);
  if (amax == 0.0f) return;
  const float inv = 1.0f / xs;
  for (int64_t b = 0; b < nb; ++b) {
    float v[16], bmax = 0.0f;
    for (int i = 0; i < 16; ++i) {
      v[i] = bf16_to_f32(hidden_row[b * 16 + i]) * inv;
      if (fabsf(v[i]) > bmax) bmax = fabsf(v[i]);
    }
    const uint8_t sc = orc_e4m3_encode(bmax / 6.0f);
    ((uint8_t*)sf_row)[b] = sc;  /* little-endian: byte b of the row */
    const float sd = orc_e4m3_decode(sc);
    if (sd == 0.0f) continue;
    const float rs = 1.0f / sd;
    for (int i = 0; i < 16; ++i) {
      const uint8_t q = orc_e2m1_encode(v[i] * rs);
      const int64_t e = b * 16 + i;
      x_row[e / 2] |= (uint8_t)(e % 2 == 0 ? q : (q << 4));
    }
  }
}

void orc_nvfp4_rows(int64_t T, int64_t K, const uint16_t* hidden, uint8_t* x, int32_t* x_sf,
                    float* x_scales) {
  const int64_t Wn = (K / 16 + 3) / 4;
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t)
    orc_nvfp4_row(K, hidden + t * K, x + t * (K / 2), x_sf + t * Wn, x_scales + t);
}

/* S6: dispatch to the batched [E, M_max, .] layout.  Routes are visited in  */
/* (token, k) order; each takes the next free slot of its expert.  A route   */
/* whose expert is full is not placed (route_slot = -1) and the function     */
/* returns 1 (capacity).  sf rows are packed UE8M0 words [., ceil(G/4)].     */
/* ------------------------------------------------------------------------ */
/* W: 4-byte words per scale row (packed UE8M0 words, or fp32 scales).     */
int orc_dispatch(int64_t T, int64_t top_k, int64_t K, const int64_t* ids, const uint8_t* x,
                 const int32_t* x_sf, int64_t W, int64_t E, int64_t M_max,
                 int32_t* expert_num_tokens, int32_t* route_slot, uint8_t* x_b, int32_t* sf_b) {
  int status = 0;
  for (int64_t e = 0; e < E; ++e) expert_num_tokens[e] = 0;
  for (int64_t t = 0; t < T; ++t) {
    for (int64_t j = 0; j < top_k; ++j) {
      int64_t id = ids[t * top_k + j];
      route_slot[t * top_k + j] = -1;
      if (id < 0) continue;
      if (id >= E) { status = 3; continue; }
      int64_t slot = expert_num_tokens[id];
      if (slot >= M_max) { status = 1; continue; }
      expert_num_tokens[id] += 1;
      route_slot[t * top_k + j] = (int32_t)slot;
      if (x_b) memcpy(x_b + (id * M_max + slot) * K, x + t * K, (size_t)K);
      if (sf_b)
        memcpy(sf_b + (id * M_max + slot) * W, x_sf + t * W, (size_t)W * sizeof(int32_t));
    }
  }
  return status;
}

/* ------------------------------------------------------------------------ */
/* S6b: contiguous layout (HummingGroupedExperts.apply: moe_permute gives    */
/* expert_offsets and the permuted rows).  Routes are visited in (token, k)  */
/* order; the routes of expert e take rows offsets[e], offsets[e] + 1, ...  */
/* where offsets[e] counts the routes to experts < e.  route_row[t, j] is    */
/* the row (-1 when unrouted).  Returns 3 on an id >= E.                     */
int orc_dispatch_contiguous(int64_t T, int64_t top_k, int64_t K, const int64_t* ids,
                            const uint8_t* x, const int32_t* x_sf, int64_t W, int64_t E,
                            int32_t* offsets, int32_t* expert_num_tokens, int32_t* route_row,
                            uint8_t* x_c, int32_t* sf_c) {
  int status = 0;
  for (int64_t e = 0; e < E; ++e) expert_num_tokens[e] = 0;
  for (int64_t r = 0; r < T * top_k; ++r) {
    const int64_t id = ids[r];
    if (id >= E) status = 3;
    if (id >= 0 && id < E) expert_num_tokens[id] += 1;
  }
  offsets[0] = 0;
  for (int64_t e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + expert_num_tokens[e];
  int32_t* filled = (int32_t*)calloc((size_t)E, sizeof(int32_t));
  for (int64_t t = 0; t < T; ++t) {
    for (int64_t j = 0; j < top_k; ++j) {
      const int64_t id = ids[t * top_k + j];
      route_row[t * top_k + j] = -1;
      if (id < 0 || id >= E) continue;
      const int64_t row = offsets[id] + filled[id];
      filled[id] += 1;
      route_row[t * top_k + j] = (int32_t)row;
      if (x_c) memcpy(x_c + row * K, x + t * K, (size_t)K);
      if (sf_c) memcpy(sf_c + row * W, x_sf + t * W, (size_t)W * sizeof(int32_t));
    }
  }
  free(filled);
  return status;
}

/* S7a: w13 GEMM + SiLU-and-mul + UE8M0 requant, for selected rows.          */
/* rows       : n_rows global row indices r = e * M_max + m                  */
/* x_b        : fp8 [E*M_max, K]; a_sf: packed UE8M0 words [E*M_max, ceil(G/4)]*/
/* w13        : fp8 [E, 2N, K]; w13_s: fp32 [E, 2N/128, K/128]               */
/* h_out      : optional bf16 bits [E*M_max, 2N] (gate columns [0,N), up     */
/*              columns [N,2N))                                              */
/* y_q, y_sf  : fp8 [E*M_max, N]; packed UE8M0 words [E*M_max, ceil(N/128/4)]*/
/* ------------------------------------------------------------------------ */
static double a_scale_of(const int32_t* sf_words, int64_t W, int64_t row, int64_t g) {
  uint32_t w = (uint32_t)sf_words[row * W + g / 4];
  int e = (int)((w >> (8 * (g % 4))) & 0xFFu);
  return ldexp(1.0, e - 127);
}

/* SiLU-and-mul of one row of bf16 h (gate [0,N), up [N,2N)) and the 1x128
 * UE8M0 requant of y along N (HummingExpertsBase.process_input with an
 * activation; the same group recipe as _quantize_fp8_groups). */
static void silu_requant_row(const double* hb, int64_t N, uint8_t* yq_row, uint32_t* ysf_row) {
  const int64_t Gn = N / 128, Wy = (Gn + 3) / 4;
  float* y = (float*)malloc(sizeof(float) * (size_t)N);
  for (int64_t n = 0; n < N; ++n) {
    double g = hb[n], u = hb[N + n];
    double silu = g / (1.0 + exp(-g));
    y[n] = (float)(silu * u);
  }
  for (int64_t w = 0; w < Wy; ++w) ysf_row[w] = 0;
  for (int64_t g = 0; g < Gn; ++g) {
    uint32_t code;
    quantize_group_f32(y + g * 128, 128, 1, yq_row + g * 128, &code, NULL);
    ysf_row[g / 4] |= (code & 0xFFu) << (8 * (g % 4));
  }
  free(y);
}

/* row_expert[i] (nullable): expert of rows[i]; NULL means rows[i] / M_max  */
/* (batched layout).                                                         */
void orc_w13_rows(int64_t n_rows, const int64_t* rows, int64_t M_max, int64_t K, int64_t N,
                  const uint8_t* x_b, const int32_t* a_sf, const uint8_t* w13,
                  const float* w13_s, uint16_t* h_out, uint8_t* y_q, int32_t* y_sf,
                  const int64_t* row_expert, int a_sf_fp32) {
  const int64_t G = K / 128, Wa = (G + 3) / 4;
  const int64_t Gn = N / 128, Wy = (Gn + 3) / 4;
  const int64_t twoN = 2 * N;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < n_rows; ++i) {
    const int64_t r = rows[i];
    const int64_t e = row_expert ? row_expert[i] : r / M_max;
    double* a = (double*)malloc(sizeof(double) * (size_t)K);
    double* hb = (double*)malloc(sizeof(double) * (size_t)twoN);
    for (int64_t k = 0; k < K; ++k)
      a[k] = (double)orc_e4m3_decode(x_b[r * K + k]) *
             (a_sf_fp32 ? (double)((const float*)a_sf)[r * G + k / 128]
                        : a_scale_of(a_sf, Wa, r, k / 128));
    for (int64_t j = 0; j < twoN; ++j) {
      const uint8_t* wrow = w13 + (e * twoN + j) * K;
      const float* srow = w13_s + (e * (twoN / 128) + j / 128) * G;
      double acc = 0.0;
      for (int64_t k = 0; k < K; ++k)
        acc += a[k] * ((double)orc_e4m3_decode(wrow[k]) * (double)srow[k / 128]);
      uint16_t hbits = orc_bf16_from_f64(acc);  /* gate_up_output is bf16 */
      if (h_out) h_out[r * twoN + j] = hbits;
      hb[j] = (double)bf16_to_f32(hbits);
    }
    silu_requant_row(hb, N, y_q + r * N, (uint32_t*)y_sf + r * Wy);
    free(a);
    free(hb);
  }
}

/* S7a second half alone: SiLU-and-mul + requant of given bf16 h rows. */
void orc_silu_requant_rows(int64_t n_rows, const int64_t* rows, int64_t N, const uint16_t* h,
                           uint8_t* y_q, int32_t* y_sf) {
  const int64_t Wy = (N / 128 + 3) / 4;
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n_rows; ++i) {
    const int64_t r = rows[i];
    double* hb = (double*)malloc(sizeof(double) * (size_t)(2 * N));
    for (int64_t j = 0; j < 2 * N; ++j) hb[j] = (double)bf16_to_f32(h[r * 2 * N + j]);
    silu_requant_row(hb, N, y_q + r * N, (uint32_t*)y_sf + r * Wy);
    free(hb);
  }
}

/* S7b: w2 GEMM for selected rows: out_b[r, c] = bf16(sum_n deq(y) deq(w2)). */
void orc_w2_rows(int64_t n_rows, const int64_t* rows, int64_t M_max, int64_t K, int64_t N,
                 const uint8_t* y_q, const int32_t* y_sf, const uint8_t* w2,
                 const float* w2_s, uint16_t* out_b, const int64_t* row_expert) {
  const int64_t Gn = N / 128, Wy = (Gn + 3) / 4;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < n_rows; ++i) {
    const int64_t r = rows[i];
    const int64_t e = row_expert ? row_expert[i] : r / M_max;
    double* a = (double*)malloc(sizeof(double) * (size_t)N);
    for (int64_t n = 0; n < N; ++n)
      a[n] = (double)orc_e4m3_decode(y_q[r * N + n]) * a_scale_of(y_sf, Wy, r, n / 128);
    for (int64_t c = 0; c < K; ++c) {
      const uint8_t* wrow = w2 + (e * K + c) * N;
      const float* srow = w2_s + (e * (K / 128) + c / 128) * Gn;
      double acc = 0.0;
      for (int64_t n = 0; n < N; ++n)
        acc += a[n] * ((double)orc_e4m3_decode(wrow[n]) * (double)srow[n / 128]);
      out_b[r * K + c] = orc_bf16_from_f64(acc);
    }
    free(a);
  }
}

/* ------------------------------------------------------------------------ */
/* S8: top-k weighted reduce back to token order.                            */
/* out[t, c] = bf16( sum_{j: slot >= 0} w[t,j] * out_b[id, slot, c] ), j     */
/* ascending; tokens without a placed route give zeros.                      */
/* num_valid (moe_fused_mul_sum's num_valid_tokens on the experts page, a   */
/* device scalar there): rows t >= num_valid are not written; a negative     */
/* value means every token.                                                  */
/* ------------------------------------------------------------------------ */
void orc_topk_reduce(int64_t T, int64_t top_k, int64_t K, int64_t M_max, const uint16_t* out_b,
                     const int64_t* ids, const int32_t* route_slot, const float* w,
                     uint16_t* out, int64_t num_valid) {
  const int64_t bound = num_valid < 0 ? T : (num_valid < T ? num_valid : T);
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < bound; ++t) {
    for (int64_t c = 0; c < K; ++c) {
      double acc = 0.0;
      for (int64_t j = 0; j < top_k; ++j) {
        int32_t s = route_slot[t * top_k + j];
        int64_t row;
        if (ids) {
          int64_t id = ids[t * top_k + j];
          if (id < 0 || s < 0) continue;
          row = id * M_max + s;
        } else {  /* contiguous layout (moe_unpermute): the slot is the row */
          if (s < 0) continue;
          row = s;
        }
        acc += (double)w[t * top_k + j] * (double)bf16_to_f32(out_b[row * K + c]);
      }
      out[t * K + c] = orc_bf16_from_f64(acc);
    }
  }
}
