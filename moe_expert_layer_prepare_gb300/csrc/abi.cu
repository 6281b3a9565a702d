// C ABI of the library: argument checks, error reporting and dispatch to the
// kernel launchers.  Every check here happens before anything is enqueued.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "common.cuh"

namespace moe_host {

static thread_local char g_last_error[512] = "";

moe_status_t set_error(moe_status_t st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return st;
}

// SM count and occupancy queries, cached per device (and per kernel and
// block size) under one lock: concurrent first calls from several host
// threads, or on several devices, all see complete entries.
static std::mutex g_query_mu;

int num_sms() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
  std::lock_guard<std::mutex> lock(g_query_mu);
  if (cached[dev] == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
      v = 152;
    cached[dev] = v;
  }
  return cached[dev];
}

// Resident blocks per SM of a kernel at a block size with no dynamic shared
// memory.  When the table is full the query is made each time.
int resident_blocks(const void* kernel, int block) {
  struct Entry {
    const void* kernel;
    int block, dev, blocks;
  };
  constexpr int kEntries = 256;
  static Entry table[kEntries] = {};
  static int used = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
  std::lock_guard<std::mutex> lock(g_query_mu);
  for (int i = 0; i < used; ++i)
    if (table[i].kernel == kernel && table[i].block == block && table[i].dev == dev)
      return table[i].blocks;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, block, 0) != cudaSuccess || n < 1)
    n = 1;
  if (used < kEntries) table[used++] = Entry{kernel, block, dev, n};
  return n;
}

size_t prepare_workspace_size(int64_t T, int64_t k, int64_t E);
moe_status_t launch_prepare(const moe_prepare_args_t* a, cudaStream_t s);
moe_status_t launch_nvfp4(const moe_nvfp4_args_t* a, cudaStream_t s);
moe_status_t launch_topk_reduce(const void* expert_out, int64_t E, int64_t M_max, int64_t K,
                                const int64_t* idx, const int32_t* slot, const float* w,
                                int64_t T, int64_t top_k, const int32_t* num_valid, void* out,
                                cudaStream_t s);
size_t experts_workspace_size(int64_t E, int64_t M_max, int64_t K, int64_t N,
                              int64_t valid_shape_m, int which);
moe_status_t launch_experts(const moe_experts_args_t* a, cudaStream_t s);

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace moe_host

using namespace moe_host;

extern "C" {

int moe_abi_version(void) { return MOE_PREP_ABI_VERSION; }

const char* moe_last_error(void) { return g_last_error; }

size_t moe_prepare_workspace_size(int64_t num_tokens, int64_t top_k, int64_t num_experts) {
  if (num_tokens < 0 || top_k < 0 || num_experts < 0) return 0;
  return prepare_workspace_size(num_tokens, top_k, num_experts);
}

moe_status_t moe_prepare_inputs(const moe_prepare_args_t* a, void* stream) {
  g_last_error[0] = '\0';
  if (a == nullptr) return set_error(MOE_ERR_INVALID_ARGUMENT, "args is NULL");
  if (a->num_tokens < 0 || a->hidden_size < 0 || a->top_k < 0)
    return set_error(MOE_ERR_INVALID_ARGUMENT, "negative size");
  if (a->num_tokens == 0) return MOE_OK;
  if (a->hidden_size % 128 != 0)
    return set_error(MOE_ERR_SHAPE, "hidden_size %lld is not a multiple of 128",
                     (long long)a->hidden_size);
  if (a->top_k < 1) return set_error(MOE_ERR_SHAPE, "top_k must be >= 1");
  if (a->sf_mode < MOE_SF_NONE || a->sf_mode > MOE_SF_FP32)
    return set_error(MOE_ERR_INVALID_ARGUMENT, "bad sf_mode %d", a->sf_mode);
  if ((a->sf_mode != MOE_SF_NONE) != (a->x_sf != nullptr))
    return set_error(MOE_ERR_INVALID_ARGUMENT, "x_sf must be given iff sf_mode != NONE");
  if (a->topk_ids_dtype != MOE_IDS_INT32 && a->topk_ids_dtype != MOE_IDS_INT64)
    return set_error(MOE_ERR_INVALID_ARGUMENT, "bad topk_ids_dtype");
  if (a->topk_weights_dtype != MOE_WEIGHTS_FP32 && a->topk_weights_dtype != MOE_WEIGHTS_BF16)
    return set_error(MOE_ERR_INVALID_ARGUMENT, "bad topk_weights_dtype");
  if (!a->hidden || !a->x || !a->topk_ids || !a->topk_weights || !a->topk_idx_out ||
      !a->topk_weights_out)
    return set_error(MOE_ERR_INVALID_ARGUMENT, "a required pointer is NULL");
  const int64_t K = a->hidden_size;
  const int64_t G = K / 128;
  if (a->hidden_stride0 < K || a->x_stride0 < K)
    return set_error(MOE_ERR_SHAPE, "row stride smaller than hidden_size");
  const int64_t x_elem = a->sf_mode == MOE_SF_NONE ? 2 : 1;
  if (!aligned16(a->hidden) || (a->hidden_stride0 * 2) % 16 != 0 || !aligned16(a->x) ||
      (a->x_stride0 * x_elem) % 16 != 0)
    return set_error(MOE_ERR_ALIGNMENT, "hidden/x rows must start on 16-byte boundaries");
  if (a->num_tokens * ((G + 3) / 4) >= ((int64_t)1 << 31))
    return set_error(MOE_ERR_UNSUPPORTED, "num_tokens * ceil(K/512) must be below 2^31");
  if (a->sf_mode == MOE_SF_UE8M0_PACKED && a->x_sf_stride1 < 1 && (G + 3) / 4 > 1)
    return set_error(MOE_ERR_SHAPE, "x_sf stride1 must be positive");
  if ((a->shared_x_sf != nullptr) != (a->shared_block_m != 0))
    return set_error(MOE_ERR_INVALID_ARGUMENT,
                     "shared_x_sf and shared_block_m must be given together");
  if (a->shared_x_sf != nullptr) {
    if (a->sf_mode != MOE_SF_UE8M0_PACKED)
      return set_error(MOE_ERR_UNSUPPORTED, "shared_x_sf requires MOE_SF_UE8M0_PACKED scales");
    if (a->shared_block_m < 0)
      return set_error(MOE_ERR_INVALID_ARGUMENT, "shared_block_m must be positive");
    const int64_t aligned = (a->shared_block_m + 127) / 128 * 128;
    const int64_t need = (a->num_tokens + a->shared_block_m - 1) / a->shared_block_m * aligned;
    if (a->shared_x_sf_rows < need)
      return set_error(MOE_ERR_SHAPE, "shared_x_sf needs %lld rows, got %lld", (long long)need,
                       (long long)a->shared_x_sf_rows);
    if (a->shared_x_sf_stride0 < 1 || (G > 1 && a->shared_x_sf_stride1 < 1))
      return set_error(MOE_ERR_SHAPE, "shared_x_sf strides must be positive");
  }
  if (a->logical_to_physical != nullptr) {
    if (a->logical_replica_count == nullptr || a->num_logical <= 0 || a->map_stride <= 0)
      return set_error(MOE_ERR_INVALID_ARGUMENT,
                       "EPLB needs logical_replica_count, num_logical and map_stride");
    if (a->expert_load != nullptr && a->num_physical <= 0)
      return set_error(MOE_ERR_INVALID_ARGUMENT, "expert_load needs num_physical > 0");
  }
  if (a->x_b != nullptr) {
    if (a->sf_mode == MOE_SF_NONE)
      return set_error(MOE_ERR_UNSUPPORTED, "dispatch requires quantised (UE8M0 or fp32) scales");
    if (a->top_k > 32)
      return set_error(MOE_ERR_UNSUPPORTED, "dispatch supports top_k <= 32");
    if (a->num_experts <= 0 || a->num_experts > 1024 || a->max_tokens_per_expert <= 0)
      return set_error(MOE_ERR_SHAPE, "dispatch needs 0 < num_experts <= 1024, M_max > 0");
    if (!a->sf_b || !a->expert_num_tokens || !a->route_slot)
      return set_error(MOE_ERR_INVALID_ARGUMENT, "dispatch needs sf_b, expert_num_tokens, route_slot");
    if (!aligned16(a->x_b))
      return set_error(MOE_ERR_ALIGNMENT, "x_b must be 16-byte aligned");
    const size_t need = prepare_workspace_size(a->num_tokens, a->top_k, a->num_experts);
    if (a->workspace == nullptr || a->workspace_bytes < need)
      return set_error(MOE_ERR_WORKSPACE, "dispatch workspace needs %zu bytes, got %zu", need,
                       a->workspace_bytes);
    if ((reinterpret_cast<uintptr_t>(a->workspace) & 255u) != 0)
      return set_error(MOE_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
    if (a->expert_offsets != nullptr &&
        a->num_tokens * a->top_k > a->num_experts * a->max_tokens_per_expert)
      return set_error(MOE_ERR_SHAPE,
                       "contiguous layout needs num_experts * max_tokens_per_expert >= %lld rows",
                       (long long)(a->num_tokens * a->top_k));
  } else if (a->expert_offsets != nullptr) {
    return set_error(MOE_ERR_INVALID_ARGUMENT, "expert_offsets needs the dispatch outputs (x_b)");
  }
  return launch_prepare(a, static_cast<cudaStream_t>(stream));
}

moe_status_t moe_prepare_nvfp4_inputs(const moe_nvfp4_args_t* a, void* stream) {
  g_last_error[0] = '\0';
  if (a == nullptr) return set_error(MOE_ERR_INVALID_ARGUMENT, "args is NULL");
  if (a->num_tokens < 0 || a->hidden_size < 0 || a->top_k < 0 || a->num_local_experts < 0)
    return set_error(MOE_ERR_INVALID_ARGUMENT, "negative size");
  if ((a->w2_global_scale == nullptr) != (a->l2_alpha == nullptr))
    return set_error(MOE_ERR_INVALID_ARGUMENT, "w2_global_scale and l2_alpha go together");
  if (a->l2_alpha != nullptr && a->num_local_experts == 0)
    return set_error(MOE_ERR_INVALID_ARGUMENT, "l2_alpha needs num_local_experts > 0");
  if (a->shared_x_dtype != MOE_SHARED_BF16 && a->shared_x_dtype != MOE_SHARED_FP8)
    return set_error(MOE_ERR_INVALID_ARGUMENT, "bad shared_x_dtype %d", a->shared_x_dtype);
  {
    // the page: shared_x_sf and shared_block_m are given exactly for an fp8 shared_x
    const bool fp8_shared = a->shared_x != nullptr && a->shared_x_dtype == MOE_SHARED_FP8;
    if (fp8_shared != (a->shared_x_sf != nullptr) ||
        (a->shared_x_sf == nullptr) != (a->shared_block_m == 0))
      return set_error(MOE_ERR_INVALID_ARGUMENT,
                       "NVFP4 staging needs shared_x_sf and shared_block_m exactly for an fp8 "
                       "shared_x");
  }
  if (a->num_tokens == 0 && a->l2_alpha == nullptr) return MOE_OK;
  if (a->hidden_size % 128 != 0)
    return set_error(MOE_ERR_SHAPE, "hidden_size %lld is not a multiple of 128",
                     (long long)a->hidden_size);
  if (a->shared_x_sf != nullptr && a->num_tokens > 0) {
    if (a->shared_block_m < 0)
      return set_error(MOE_ERR_INVALID_ARGUMENT, "shared_block_m must be positive");
    const int64_t aligned = (a->shared_block_m + 127) / 128 * 128;
    const int64_t need = (a->num_tokens + a->shared_block_m - 1) / a->shared_block_m * aligned;
    if (a->shared_x_sf_rows < need)
      return set_error(MOE_ERR_SHAPE, "shared_x_sf needs %lld rows, got %lld", (long long)need,
                       (long long)a->shared_x_sf_rows);
    if (a->shared_x_sf_stride0 < 1 || (a->hidden_size > 128 && a->shared_x_sf_stride1 < 1))
      return set_error(MOE_ERR_SHAPE, "shared_x_sf strides must be positive");
  }
  if (a->num_tokens > 0) {
    if (a->top_k < 1) return set_error(MOE_ERR_SHAPE, "top_k must be >= 1");
    if (a->topk_ids_dtype != MOE_IDS_INT32 && a->topk_ids_dtype != MOE_IDS_INT64)
      return set_error(MOE_ERR_INVALID_ARGUMENT, "bad topk_ids_dtype");
    if (a->topk_weights_dtype != MOE_WEIGHTS_FP32 && a->topk_weights_dtype != MOE_WEIGHTS_BF16)
      return set_error(MOE_ERR_INVALID_ARGUMENT, "bad topk_weights_dtype");
    if (!a->hidden || !a->x || !a->x_sf || !a->x_scales || !a->topk_ids || !a->topk_weights ||
        !a->topk_idx_out || !a->topk_weights_out)
      return set_error(MOE_ERR_INVALID_ARGUMENT, "a required pointer is NULL");
    const int64_t K = a->hidden_size;
    if (a->hidden_stride0 < K || a->x_stride0 < K / 2 || a->x_sf_stride0 < K / 64 ||
        (a->shared_x != nullptr && a->shared_x_stride0 < K))
      return set_error(MOE_ERR_SHAPE, "row stride smaller than the row");
    const int64_t shared_elem = a->shared_x_dtype == MOE_SHARED_FP8 ? 1 : 2;
    if (!aligned16(a->hidden) || (a->hidden_stride0 * 2) % 16 != 0 ||
        (reinterpret_cast<uintptr_t>(a->x) & 3u) != 0 || a->x_stride0 % 4 != 0 ||
        (a->shared_x != nullptr &&
         (!aligned16(a->shared_x) || (a->shared_x_stride0 * shared_elem) % 16 != 0)))
      return set_error(MOE_ERR_ALIGNMENT, "hidden/shared_x rows must start on 16-byte and x "
                                          "rows on 4-byte boundaries");
    if (a->logical_to_physical != nullptr &&
        (a->logical_replica_count == nullptr || a->num_logical <= 0 || a->map_stride <= 0))
      return set_error(MOE_ERR_INVALID_ARGUMENT,
                       "EPLB needs logical_replica_count, num_logical and map_stride");
    if (a->expert_load != nullptr && a->num_physical <= 0)
      return set_error(MOE_ERR_INVALID_ARGUMENT, "expert_load needs num_physical > 0");
  }
  return launch_nvfp4(a, static_cast<cudaStream_t>(stream));
}

size_t moe_batched_experts_workspace_size(int64_t num_experts, int64_t max_tokens_per_expert,
                                          int64_t hidden_size, int64_t intermediate_size,
                                          int64_t valid_shape_m, int which) {
  if (num_experts <= 0 || max_tokens_per_expert <= 0 || hidden_size <= 0 ||
      intermediate_size <= 0)
    return 0;
  return experts_workspace_size(num_experts, max_tokens_per_expert, hidden_size,
                                intermediate_size, valid_shape_m, which);
}

moe_status_t moe_batched_experts(const moe_experts_args_t* a, void* stream) {
  g_last_error[0] = '\0';
  if (a == nullptr) return set_error(MOE_ERR_INVALID_ARGUMENT, "args is NULL");
  if (a->num_experts <= 0 || a->max_tokens_per_expert <= 0 || a->hidden_size <= 0 ||
      a->intermediate_size <= 0)
    return set_error(MOE_ERR_INVALID_ARGUMENT, "sizes must be positive");
  if (a->hidden_size % 128 != 0 || a->intermediate_size % 128 != 0)
    return set_error(MOE_ERR_SHAPE, "hidden_size and intermediate_size must be multiples of 128");
  if (a->activation != MOE_ACT_SILU)
    return set_error(MOE_ERR_UNSUPPORTED, "only SiLU-and-mul is implemented");
  if (a->a_scale_mode != MOE_SF_UE8M0_PACKED && a->a_scale_mode != MOE_SF_FP32)
    return set_error(MOE_ERR_UNSUPPORTED,
                     "activation scales must be MOE_SF_UE8M0_PACKED or MOE_SF_FP32");
  const int stages = a->stages == 0 ? MOE_STAGE_ALL : a->stages;
  if (stages < 1 || stages > 3) return set_error(MOE_ERR_INVALID_ARGUMENT, "bad stages mask");
  if (!a->expert_num_tokens) return set_error(MOE_ERR_INVALID_ARGUMENT, "expert_num_tokens is NULL");
  if (stages & MOE_STAGE_W13) {
    if (!a->hidden || !a->a_scale || !a->w13 || !a->w13_scale)
      return set_error(MOE_ERR_INVALID_ARGUMENT, "w13 stage needs hidden, a_scale, w13, w13_scale");
    if (!aligned16(a->hidden) || !aligned16(a->w13))
      return set_error(MOE_ERR_ALIGNMENT, "hidden and w13 must be 16-byte aligned");
  }
  if (stages & MOE_STAGE_W2) {
    if (!a->output || !a->w2 || !a->w2_scale)
      return set_error(MOE_ERR_INVALID_ARGUMENT, "w2 stage needs output, w2, w2_scale");
    if (!aligned16(a->w2) || !aligned16(a->output))
      return set_error(MOE_ERR_ALIGNMENT, "w2 and output must be 16-byte aligned");
    if (stages == MOE_STAGE_W2 && (!a->inter_q || !a->inter_sf))
      return set_error(MOE_ERR_INVALID_ARGUMENT, "the w2 stage alone needs inter_q and inter_sf");
  }
  if ((a->inter_q == nullptr) != (a->inter_sf == nullptr))
    return set_error(MOE_ERR_INVALID_ARGUMENT, "give both inter_q and inter_sf or neither");
  if (a->inter_q && !aligned16(a->inter_q))
    return set_error(MOE_ERR_ALIGNMENT, "inter_q must be 16-byte aligned");
  const int64_t E = a->num_experts, M = a->max_tokens_per_expert;
  const int64_t K = a->hidden_size, N = a->intermediate_size;
  if (a->inter_q == nullptr) {
    const size_t need = experts_workspace_size(E, M, K, N, a->valid_shape_m, 13);
    if (!a->workspace13 || a->workspace13_bytes < need)
      return set_error(MOE_ERR_WORKSPACE, "workspace13 needs %zu bytes, got %zu", need,
                       a->workspace13_bytes);
    if ((reinterpret_cast<uintptr_t>(a->workspace13) & 255u) != 0)
      return set_error(MOE_ERR_ALIGNMENT, "workspace13 must be 256-byte aligned");
  }
  if (stages & MOE_STAGE_W2) {
    const size_t need2 = experts_workspace_size(E, M, K, N, a->valid_shape_m, 2);
    if (need2 > 0 && (!a->workspace2 || a->workspace2_bytes < need2))
      return set_error(MOE_ERR_WORKSPACE, "workspace2 needs %zu bytes, got %zu", need2,
                       a->workspace2_bytes);
    if (need2 > 0 && (reinterpret_cast<uintptr_t>(a->workspace2) & 255u) != 0)
      return set_error(MOE_ERR_ALIGNMENT, "workspace2 must be 256-byte aligned");
  }
  return launch_experts(a, static_cast<cudaStream_t>(stream));
}

moe_status_t moe_topk_reduce(const void* expert_out, int64_t num_experts,
                             int64_t max_tokens_per_expert, int64_t hidden_size,
                             const int64_t* topk_idx, const int32_t* route_slot,
                             const float* topk_weights, int64_t num_tokens, int64_t top_k,
                             const int32_t* num_valid_tokens, void* out, void* stream) {
  g_last_error[0] = '\0';
  if (num_tokens < 0 || top_k < 0 || hidden_size < 0)
    return set_error(MOE_ERR_INVALID_ARGUMENT, "negative size");
  if (num_tokens == 0 || hidden_size == 0) return MOE_OK;
  if (num_experts <= 0 || max_tokens_per_expert <= 0)
    return set_error(MOE_ERR_INVALID_ARGUMENT, "num_experts and max_tokens_per_expert must be positive");
  if (hidden_size % 8 != 0) return set_error(MOE_ERR_SHAPE, "hidden_size must be a multiple of 8");
  if (num_tokens * ((hidden_size + 255) / 256) >= ((int64_t)1 << 31))
    return set_error(MOE_ERR_UNSUPPORTED, "num_tokens * ceil(K/256) must be below 2^31");
  // topk_idx == NULL: route_slot holds rows of expert_out (contiguous layout)
  if (!expert_out || !out || (top_k > 0 && (!route_slot || !topk_weights)))
    return set_error(MOE_ERR_INVALID_ARGUMENT, "a required pointer is NULL");
  if (!aligned16(expert_out) || !aligned16(out))
    return set_error(MOE_ERR_ALIGNMENT, "expert_out and out must be 16-byte aligned");
  return launch_topk_reduce(expert_out, num_experts, max_tokens_per_expert, hidden_size,
                            topk_idx, route_slot, topk_weights, num_tokens, top_k,
                            num_valid_tokens, out, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
