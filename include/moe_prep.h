/*
 * moe_prep.h -- C ABI of the GB300 (sm_103a) batched grouped-masked block-FP8
 * MoE expert forward.
 *
 * Three entry points make up the path:
 *
 *   moe_prepare_inputs   input staging: bf16 -> fp8 e4m3 with 1x128 UE8M0
 *                        scales, top-k repack (int64 ids, fp32 weights),
 *                        EPLB replica map, and optionally the dispatch into
 *                        the batched [experts, max_tokens, K] layout.
 *   moe_batched_experts  w13 gate_up GEMM masked by expert_num_tokens, fused
 *                        SiLU-and-mul + FP8 requant, w2 down GEMM.
 *   moe_topk_reduce      top-k weighted sum back to token order.
 *
 * Conventions shared by every call
 *   - All tensor pointers are DEVICE pointers unless stated otherwise; every
 *     output buffer is allocated by the caller; the library never allocates
 *     device memory.
 *   - Strides are in ELEMENTS of the tensor's own dtype.
 *   - `stream` is a cudaStream_t passed as void*.  Work is enqueued
 *     asynchronously; nothing synchronises the host.
 *   - Host-checkable problems return a moe_status_t before anything is
 *     enqueued; moe_last_error() then holds a message (thread-local).
 *   - Problems only the device can see (an expert receiving more routes than
 *     it has rows, a routed id outside [0, num_experts), a GEMM wait that
 *     timed out) are OR-ed into *device_status (MOE_DEV_* bits) when the
 *     caller passes one.  Kernels never trap.
 */
#ifndef MOE_PREP_H
#define MOE_PREP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_PREP_ABI_VERSION 3

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARGUMENT = 1, /* NULL where required, negative size, bad enum */
  MOE_ERR_SHAPE = 2,            /* a shape rule of the pages is broken */
  MOE_ERR_UNSUPPORTED = 3,      /* a combination this library does not implement */
  MOE_ERR_ALIGNMENT = 4,        /* pointer/stride alignment needed by vector or TMA access */
  MOE_ERR_WORKSPACE = 5,        /* workspace missing or smaller than the size query */
  MOE_ERR_CUDA = 6              /* a CUDA runtime call failed */
} moe_status_t;

/* Device status bits (OR-ed into *device_status). */
#define MOE_DEV_CAPACITY 1u   /* an expert got more than max_tokens_per_expert routes */
#define MOE_DEV_BAD_EXPERT 2u /* routed id >= num_experts / num_logical, or bad EPLB entry */
#define MOE_DEV_TIMEOUT 4u    /* a bounded pipeline wait inside a GEMM expired */

typedef enum moe_sf_mode {
  MOE_SF_NONE = 0,         /* no quantisation: x receives a bf16 copy of hidden */
  MOE_SF_UE8M0_PACKED = 1, /* x_sf int32 [T, ceil(G/4)]: group g is byte g%4 of word g/4 */
  MOE_SF_FP32 = 2          /* x_sf fp32 [T, G]: the group scale amax/448 itself */
} moe_sf_mode_t;

typedef enum moe_ids_dtype { MOE_IDS_INT32 = 0, MOE_IDS_INT64 = 1 } moe_ids_dtype_t;
typedef enum moe_weights_dtype { MOE_WEIGHTS_FP32 = 0, MOE_WEIGHTS_BF16 = 1 } moe_weights_dtype_t;
typedef enum moe_activation { MOE_ACT_SILU = 0 } moe_activation_t;
typedef enum moe_shared_dtype { MOE_SHARED_BF16 = 0, MOE_SHARED_FP8 = 1 } moe_shared_dtype_t;

/* Stage mask of moe_batched_experts. */
#define MOE_STAGE_W13 1
#define MOE_STAGE_W2 2
#define MOE_STAGE_ALL 3

/* ------------------------------------------------------------------------ */
/* moe_prepare_inputs                                                        */
/*                                                                           */
/* Defined by prepare_megamoe_inputs, _quantize_fp8_groups, _pack_bytes,     */
/* _store_topk and _eplb_kernel_args on the page                             */
/* "vllm.model_executor.layers.fused_moe.prepare_megamoe", and, for the      */
/* optional dispatch, by the batched activation format of                    */
/* BatchedHummingGroupedExperts ("...fused_moe.experts.fused_humming_moe":   */
/* hidden_states [E, max_tokens, K] with expert_tokens_meta.expert_num_tokens).*/
/*                                                                           */
/* Per token t and 1x128 group g of hidden (G = K/128 groups):               */
/*   amax = max(max|x|, 1e-4); s = amax / 448 (fp32);                        */
/*   UE8M0: e = expfield(s) + (mantissa(s) != 0), clamped to [1, 254],       */
/*          qs = 2^(e-127);  FP32: qs = s;                                    */
/*   x[t, i] = e4m3_rn_satfinite(hidden[t, i] * (1 / qs)).                   */
/* Top-k: topk_idx_out = int64(topk_ids), topk_weights_out = fp32(weights);  */
/* padding tokens (is_padding[t] != 0) get id -1 and weight 0.               */
/* EPLB (when logical_to_physical != NULL) maps a routed logical id l to     */
/* logical_to_physical[l * map_stride + (t mod logical_replica_count[l])]    */
/* and, when *should_record != 0 and t < *num_unpadded_tokens, adds 1 to     */
/* expert_load[physical id].                                                 */
/* Dispatch (when x_b != NULL; UE8M0 or FP32 scales): routes are            */
/* placed in (token, k) order; route (t, j) with id e takes slot s, the      */
/* number of earlier routes to e, and x_b[e, s, :] = x[t, :],                */
/* sf_b[e, s, :] = x_sf[t, :], route_slot[t, j] = s (-1 when unrouted or     */
/* when s >= max_tokens_per_expert, which also sets MOE_DEV_CAPACITY),       */
/* expert_num_tokens[e] = min(#routes to e, max_tokens_per_expert).          */
/* Contiguous layout (when expert_offsets != NULL; the expert_offsets /     */
/* moe_permute layout of HummingGroupedExperts.apply on the experts page):  */
/* no per-expert capacity; the routes of expert e fill rows                 */
/* [expert_offsets[e], expert_offsets[e+1]) of x_b / sf_b in the same       */
/* (token, k) order, expert_offsets[e] = #routes to experts < e,            */
/* expert_offsets[E] = #routes, route_slot[t, j] = the row (not the slot)   */
/* and expert_num_tokens[e] the full count.  x_b / sf_b hold                */
/* E * max_tokens_per_expert rows, which must be >= T * k (else SHAPE).     */
/*                                                                           */
/* Shared-expert scale pages (when shared_x_sf != NULL; defined by the      */
/* shared_x_sf / shared_block_m arguments of prepare_megamoe_inputs and by   */
/* _shared_sf_row on the same page; requires MOE_SF_UE8M0_PACKED): the      */
/* exponent byte e of group g of token t is also written to                  */
/*   shared_x_sf[row(t) * shared_x_sf_stride0 + g * shared_x_sf_stride1],   */
/* one uint8 per (row, group) (reading: the page's UE8M0 scale element is    */
/* its exponent byte).  With B = shared_block_m, A = ceil(B/128)*128,        */
/* b = t / B and m = t % B:                                                  */
/*   row(t) = b*A + (m/128)*128 + (m%32)*4 + (m%128)/32,                     */
/* i.e. each 128-row page interleaves its four 32-token quarters row by row */
/* (the MN-major layout a tcgen05.cp of the scales expects).  Rows that no   */
/* token maps to are left untouched.  The buffer must hold at least         */
/* ceil(T/B)*A rows (shared_x_sf_rows), else SHAPE.                          */
/*                                                                           */
/* Errors: T == 0 -> MOE_OK, nothing enqueued.  K % 128 != 0 -> SHAPE.       */
/* x_sf given iff sf_mode != NONE, else INVALID_ARGUMENT.  top_k < 1 ->       */
/* SHAPE.  hidden / x rows must start on 16-byte boundaries (ALIGNMENT).     */
/* Dispatch needs workspace of moe_prepare_workspace_size() bytes (WORKSPACE)*/
/* and top_k <= 32 (UNSUPPORTED).                                            */
/* ------------------------------------------------------------------------ */
typedef struct moe_prepare_args {
  int64_t num_tokens;  /* T >= 0 */
  int64_t hidden_size; /* K, multiple of 128 */
  int64_t top_k;       /* k >= 1 */

  const void* hidden; /* bf16 [T, K], inner stride 1 */
  int64_t hidden_stride0;
  const void* topk_ids; /* int32 or int64 [T, k] */
  int32_t topk_ids_dtype;
  int64_t topk_ids_stride0, topk_ids_stride1;
  const void* topk_weights; /* fp32 or bf16 [T, k] */
  int32_t topk_weights_dtype;
  int64_t topk_weights_stride0, topk_weights_stride1;
  const uint8_t* is_padding; /* nullable; [T], nonzero = padding */
  int64_t is_padding_stride0;

  void* x; /* fp8 e4m3 [T, K] (bf16 when sf_mode == MOE_SF_NONE), inner stride 1 */
  int64_t x_stride0;
  void* x_sf; /* NULL iff sf_mode == MOE_SF_NONE */
  int32_t sf_mode;
  int64_t x_sf_stride0, x_sf_stride1;
  uint8_t* shared_x_sf;    /* nullable; UE8M0 exponent bytes [shared_x_sf_rows, K/128] */
  int64_t shared_x_sf_stride0, shared_x_sf_stride1;
  int64_t shared_x_sf_rows; /* rows of shared_x_sf */
  int64_t shared_block_m;   /* > 0 iff shared_x_sf != NULL */
  int64_t* topk_idx_out; /* int64 [T, k] */
  int64_t topk_idx_out_stride0, topk_idx_out_stride1;
  float* topk_weights_out; /* fp32 [T, k] */
  int64_t topk_weights_out_stride0, topk_weights_out_stride1;

  /* EPLB: all NULL / 0 leaves ids unmapped. */
  const int32_t* logical_to_physical; /* [num_logical, map_stride] */
  int64_t num_logical, map_stride;
  const int32_t* logical_replica_count; /* [num_logical], each >= 1 */
  int32_t* expert_load;                 /* nullable; [num_physical] */
  int64_t num_physical;
  const uint8_t* should_record;       /* nullable device scalar; NULL = never record */
  const int32_t* num_unpadded_tokens; /* nullable device scalar; NULL = T */

  /* Optional dispatch into the batched layout (x_b == NULL disables it). */
  int64_t num_experts;           /* E */
  int64_t max_tokens_per_expert; /* M_max */
  void* x_b;                     /* fp8 [E, M_max, K] */
  void* sf_b;                    /* int32 [E, M_max, ceil(G/4)] packed UE8M0, or fp32 [E, M_max, G] */
  int32_t* expert_num_tokens;    /* int32 [E] */
  int32_t* route_slot;           /* int32 [T, k], contiguous */
  int32_t* expert_offsets;       /* nullable int32 [E + 1]: contiguous layout */
  void* workspace;               /* moe_prepare_workspace_size() bytes */
  size_t workspace_bytes;

  uint32_t* device_status; /* nullable; MOE_DEV_* bits are OR-ed in */
} moe_prepare_args_t;

moe_status_t moe_prepare_inputs(const moe_prepare_args_t* args, void* stream);

/* Bytes of workspace the dispatch of moe_prepare_inputs needs. */
size_t moe_prepare_workspace_size(int64_t num_tokens, int64_t top_k, int64_t num_experts);

/* ------------------------------------------------------------------------ */
/* moe_prepare_nvfp4_inputs                                                  */
/*                                                                           */
/* Defined by prepare_megamoe_nvfp4_inputs (kNvfp4DynamicToken) on the page  */
/* "vllm.model_executor.layers.fused_moe.prepare_megamoe": each token is     */
/* scaled by its own fp32 x_scales (row amax / 2688) and quantised to E2M1   */
/* with one E4M3 scale per 16 values.  The kernel body is not on the page;  */
/* this library computes, in fp32 with IEEE roundings, per token t:          */
/*   xs = amax / 2688;  v_i = x_i * (1 / xs);                                */
/*   per 16 values: s = e4m3_rn_satfinite(max|v_i| / 6),                     */
/*                  q_i = e2m1_rn_satfinite(v_i * (1 / dec(s)));             */
/* amax == 0 gives xs = 0 and zero codes and scales; a block whose scale    */
/* rounds to 0 gets zero codes.  x: uint8 [T, K/2], value 2i in the low     */
/* nibble of byte i; x_sf: int32 [T, K/64], block b's E4M3 byte at byte     */
/* b % 4 of word b / 4; x_scales: fp32 [T].                                  */
/* Routing outputs (topk_idx_out, topk_weights_out, EPLB map and load) are  */
/* exactly those of moe_prepare_inputs.  Shared-expert input (the page's    */
/* shared_x, nullable), by shared_x_dtype:                                   */
/*   MOE_SHARED_BF16: bf16 [T, K], a copy of the hidden rows;                */
/*   MOE_SHARED_FP8 (MXFP8 with shared_x_sf): fp8 e4m3 [T, K], the hidden    */
/*     rows quantised exactly as moe_prepare_inputs quantises x (1x128        */
/*     groups, UE8M0 scales), and each group's exponent byte written to      */
/*     shared_x_sf at row(t) of the shared-expert pages of shared_block_m     */
/*     (the same layout and row rule as moe_prepare_inputs' shared_x_sf).    */
/* shared_x_sf and shared_block_m are given exactly for an fp8 shared_x      */
/* (else INVALID_ARGUMENT, as the page raises); shared_x_sf must hold         */
/* ceil(T/B)*A rows (SHAPE).                                                 */
/* l2_alpha[e] = w2_global_scale[e] * l2_activation_scale for e <            */
/* num_local_experts, written even when T == 0 (both NULL or both given).    */
/* Errors: K % 128 != 0 -> SHAPE; rows of hidden, x, shared_x not 16-byte    */
/* aligned -> ALIGNMENT; w2_global_scale without l2_alpha -> INVALID.        */
/* ------------------------------------------------------------------------ */
typedef struct moe_nvfp4_args {
  int64_t num_tokens, hidden_size, top_k;
  const void* hidden; /* bf16 [T, K] */
  int64_t hidden_stride0;
  const void* topk_ids;
  int32_t topk_ids_dtype;
  int64_t topk_ids_stride0, topk_ids_stride1;
  const void* topk_weights;
  int32_t topk_weights_dtype;
  int64_t topk_weights_stride0, topk_weights_stride1;
  const uint8_t* is_padding; /* nullable */
  int64_t is_padding_stride0;
  uint8_t* x; /* E2M1 pairs [T, K/2] */
  int64_t x_stride0;
  int32_t* x_sf; /* packed E4M3 block scales [T, K/64] */
  int64_t x_sf_stride0;
  float* x_scales; /* [T] */
  void* shared_x;  /* nullable: bf16 [T, K] copy, or fp8 [T, K] (shared_x_dtype) */
  int64_t shared_x_stride0;
  int32_t shared_x_dtype;    /* MOE_SHARED_BF16 or MOE_SHARED_FP8 */
  uint8_t* shared_x_sf;      /* fp8 shared_x only: UE8M0 bytes [shared_x_sf_rows, K/128] */
  int64_t shared_x_sf_stride0, shared_x_sf_stride1;
  int64_t shared_x_sf_rows;
  int64_t shared_block_m;    /* > 0 iff shared_x_sf != NULL */
  int64_t* topk_idx_out;
  int64_t topk_idx_out_stride0, topk_idx_out_stride1;
  float* topk_weights_out;
  int64_t topk_weights_out_stride0, topk_weights_out_stride1;
  const int32_t* logical_to_physical; /* EPLB, as in moe_prepare_args_t */
  int64_t num_logical, map_stride;
  const int32_t* logical_replica_count;
  int32_t* expert_load;
  int64_t num_physical;
  const uint8_t* should_record;
  const int32_t* num_unpadded_tokens;
  const float* w2_global_scale; /* nullable [num_local_experts] */
  float* l2_alpha;              /* nullable [num_local_experts] */
  int64_t num_local_experts;
  float l2_activation_scale;
  uint32_t* device_status;
} moe_nvfp4_args_t;

moe_status_t moe_prepare_nvfp4_inputs(const moe_nvfp4_args_t* args, void* stream);

/* ------------------------------------------------------------------------ */
/* moe_prepare_inputs_noalloc                                                */
/*                                                                           */
/* No counterpart on the pages: an addition of this library for callers that */
/* cannot allocate device memory -- a plugin that is handed only its input   */
/* and output buffers, code running under a CUDA graph capture where its      */
/* framework forbids allocation, or a process held to a fixed device-memory  */
/* budget that must never call cudaMalloc (which can also synchronise the    */
/* device).                                                                  */
/*                                                                           */
/* Same arguments, checks and results as moe_prepare_inputs, except that the */
/* dispatch scratch comes from a fixed array of                              */
/* MOE_PREPARE_NOALLOC_SCRATCH_BYTES bytes inside the library (present on    */
/* every GPU that loads it, until the process exits); args->workspace and    */
/* args->workspace_bytes are ignored.  A problem whose                       */
/* moe_prepare_workspace_size() exceeds that size returns                    */
/* MOE_ERR_WORKSPACE before anything is enqueued.  Nothing is allocated: no  */
/* cudaMalloc/cudaFree or allocating library call.  The array's device       */
/* address is looked up on the first call made with a device current, so    */
/* make that first call before any stream capture (it is looked up again     */
/* when the device's context has changed, e.g. after cudaDeviceReset).       */
/* Every call on a device shares the one array and finds the previous call's */
/* contents there (each call clears what must start at zero); calls that may */
/* overlap on the GPU race on it and must be serialised by the caller.       */
/* ------------------------------------------------------------------------ */
#define MOE_PREPARE_NOALLOC_SCRATCH_BYTES (4u << 20)

moe_status_t moe_prepare_inputs_noalloc(const moe_prepare_args_t* args, void* stream);

/* ------------------------------------------------------------------------ */
/* moe_batched_experts                                                       */
/*                                                                           */
/* Defined by BatchedHummingGroupedExperts.apply and                         */
/* HummingExpertsBase.process_input / humming_forward / get_buffer_metas on  */
/* the page "vllm.model_executor.layers.fused_moe.experts.fused_humming_moe" */
/* (GROUPED_MASKED layout, block-FP8 input pre-quantised before dispatch,    */
/* apply_router_weight_on_input false).  For each expert e and each row      */
/* m < expert_num_tokens[e] (G = K/128, Gn = N/128):                          */
/*   h[n]   = sum_k deq(x_b[e,m,k]) * w13[e,n,k] * w13_scale[e,n/128,k/128]  */
/*            for n in [0, 2N); deq(x) = x * 2^(sf - 127) per 1x128 group;    */
/*            columns [0, N) are gate, [N, 2N) up; h is rounded to bf16.      */
/*   y[n]   = silu(h[n]) * h[N+n], silu(g) = g / (1 + exp(-g)), n < N          */
/*   y is requantised to fp8 e4m3 in 1x128 UE8M0 groups (same recipe as      */
/*   moe_prepare_inputs) into inter_q / inter_sf.                             */
/*   output[e,m,c] = bf16( sum_n deq(y_q[m,n]) * w2[e,c,n] * w2_scale[e,c/128,n/128] ).*/
/* Rows m >= expert_num_tokens[e] of output (and of inter_q) are not written.*/
/* Accumulation is fp32; weight block scales are applied per 128-wide K      */
/* slab in fp32.                                                              */
/*                                                                           */
/* Layouts: x_b [E*M_max, K] fp8, a_scale int32 [E*M_max, ceil(G/4)] packed  */
/* UE8M0 (a_scale_mode MOE_SF_UE8M0_PACKED) or fp32 [E*M_max, G] with       */
/* deq(x) = x * a_scale[row, k/128] (MOE_SF_FP32: the fp32 a1q_scale        */
/* [M, K/128] contract of process_input / get_buffer_metas; the requantised */
/* w2 input stays 1x128 UE8M0), w13 [E, 2N, K] fp8 K-major,                  */
/* w13_scale fp32 [E, 2N/128, G], w2 [E, K, N] fp8 N-major, w2_scale fp32     */
/* [E, K/128, Gn], output bf16 [E, M_max, K].  All contiguous.  Base pointers*/
/* of x_b, w13, w2, inter_q must be 16-byte aligned.                          */
/* inter_q fp8 [E*M_max, N] and inter_sf int32 [E*M_max, ceil(Gn/4)] may be  */
/* NULL, in which case they are carved from workspace13.  With stages ==     */
/* MOE_STAGE_W2 the caller supplies them (the w2 stage alone).               */
/* Contiguous layout (expert_offsets != NULL, [E+1] as written by           */
/* moe_prepare_inputs; HummingGroupedExperts.apply with expert_layout =     */
/* expert_offsets): expert e owns rows [expert_offsets[e],                  */
/* expert_offsets[e+1]) of x_b / a_scale / inter_q / inter_sf / output,     */
/* which are still E*M_max rows long (expert_offsets[E] <= E*M_max), and     */
/* its row count is not capped by M_max.                                     */
/* workspace2 holds split-K partials and tile counters.  It must be zero-    */
/* filled once when allocated; every call leaves its counters at zero again   */
/* (after a MOE_DEV_TIMEOUT, zero it before reuse).                           */
/* Errors: K % 128, N % 128 -> SHAPE; activation != SILU, a_scale_mode not   */
/* UE8M0_PACKED or FP32 -> UNSUPPORTED; short workspaces -> WORKSPACE.       */
/* ------------------------------------------------------------------------ */
typedef struct moe_experts_args {
  int64_t num_experts;           /* E */
  int64_t max_tokens_per_expert; /* M_max */
  int64_t hidden_size;           /* K, multiple of 128 */
  int64_t intermediate_size;     /* N, multiple of 128 */
  int32_t activation;            /* MOE_ACT_SILU */
  int32_t stages;                /* MOE_STAGE_* mask; 0 means MOE_STAGE_ALL */

  void* output;                       /* bf16 [E, M_max, K] */
  const void* hidden;                 /* fp8 [E*M_max, K] */
  const void* a_scale;                /* int32 [E*M_max, ceil(G/4)] */
  int32_t a_scale_mode;               /* MOE_SF_UE8M0_PACKED */
  const void* w13;                    /* fp8 [E, 2N, K] */
  const float* w13_scale;             /* [E, 2N/128, K/128] */
  const void* w2;                     /* fp8 [E, K, N] */
  const float* w2_scale;              /* [E, K/128, N/128] */
  const int32_t* expert_num_tokens;   /* [E] */
  const int32_t* expert_offsets;      /* nullable [E+1]: contiguous layout */

  void* inter_q;   /* nullable: fp8 [E*M_max, N] */
  void* inter_sf;  /* nullable: int32 [E*M_max, ceil(Gn/4)] */
  void* workspace13;
  size_t workspace13_bytes;
  void* workspace2;
  size_t workspace2_bytes;
  int64_t valid_shape_m; /* tuning hint: the routed rows this call expects, the     */
                         /* pages' estimate_local_valid_shape_m (T * k, scaled by   */
                         /* local / global experts); <= 0: this call has no token   */
                         /* count, so it assumes every row of the layout (E * M_max) */
  void* gate_up_dump;    /* nullable: bf16 [E*M_max, 2N] copy of h (debug/parity) */
  uint32_t* device_status;
} moe_experts_args_t;

moe_status_t moe_batched_experts(const moe_experts_args_t* args, void* stream);

/* Workspace bytes: which = 13 (workspace13: inter_q + inter_sf) or 2
 * (workspace2: split-K partials + tile counters for this valid_shape_m). */
size_t moe_batched_experts_workspace_size(int64_t num_experts, int64_t max_tokens_per_expert,
                                          int64_t hidden_size, int64_t intermediate_size,
                                          int64_t valid_shape_m, int which);

/* ------------------------------------------------------------------------ */
/* moe_topk_reduce                                                           */
/*                                                                           */
/* Defined by the finalize step of BatchedHummingGroupedExperts              */
/* (finalize_weight_and_reduce_impl -> TopKWeightAndReduceDelegate) and the  */
/* weighted top-k sum of moe_fused_mul_sum in HummingIndexedExperts.apply     */
/* ("...fused_moe.experts.fused_humming_moe"):                               */
/*   out[t, c] = bf16( sum_{j < k, idx[t,j] >= 0, slot[t,j] >= 0}            */
/*                     w[t,j] * expert_out[idx[t,j], slot[t,j], c] )          */
/* summed in fp32 in ascending j; tokens without a placed route get 0.       */
/* expert_out bf16 [E, M_max, K]; topk_idx int64 [T, k]; route_slot int32    */
/* [T, k]; topk_weights fp32 [T, k]; out bf16 [T, K]; all contiguous; the    */
/* expert_out and out base pointers 16-byte aligned; K % 8 == 0.             */
/* Contiguous layout (moe_unpermute of HummingGroupedExperts.apply): with    */
/* topk_idx == NULL, route_slot[t, j] is the row of expert_out itself (-1 =  */
/* unplaced), rows < num_experts * max_tokens_per_expert.                    */
/* num_valid_tokens (nullable DEVICE int32 scalar; the num_valid_tokens of   */
/* moe_fused_mul_sum in HummingIndexedExperts.apply): only tokens           */
/* t < *num_valid_tokens are written, rows past it are left untouched (a     */
/* negative value writes none).  The launch is sized by num_tokens, so a     */
/* call captured in a CUDA graph with the largest batch serves every smaller */
/* batch by updating the scalar.  NULL writes all num_tokens rows.           */
/* ------------------------------------------------------------------------ */
moe_status_t moe_topk_reduce(const void* expert_out, int64_t num_experts,
                             int64_t max_tokens_per_expert, int64_t hidden_size,
                             const int64_t* topk_idx, const int32_t* route_slot,
                             const float* topk_weights, int64_t num_tokens, int64_t top_k,
                             const int32_t* num_valid_tokens, void* out, void* stream);

/* ------------------------------------------------------------------------ */
/* Utilities                                                                 */
/* ------------------------------------------------------------------------ */
int moe_abi_version(void);
/* Message of the last host-side error on this thread ("" if none). */
const char* moe_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_PREP_H */
