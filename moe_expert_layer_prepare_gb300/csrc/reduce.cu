// Top-k weighted reduce back to token order.
//
// Follows the finalize step of BatchedHummingGroupedExperts
// (TopKWeightAndReduceDelegate) and the weighted top-k sum of
// moe_fused_mul_sum in HummingIndexedExperts.apply
// ("vllm.model_executor.layers.fused_moe.experts.fused_humming_moe").
//
// One warp per (token, 256-column chunk); each lane owns 8 columns (16 bytes).
// The routes' rows and weights are resolved once per warp (one lane per
// route) and the routed expert rows are read eight at a time with streaming
// 16-byte loads, then weighted in fp32 and accumulated in ascending j; one
// bf16 rounding at the end.  HBM-bound: each routed row is read once, each output row
// written once.  An optional device scalar bounds the tokens written
// (moe_fused_mul_sum's num_valid_tokens), so that one launch configuration,
// captured in a graph, serves every smaller batch.
#include "common.cuh"

namespace moe {

struct ReduceParams {
  const uint16_t* expert_out;  // bf16 [E*M_max, K]
  int64_t E, M_max, K;
  const int64_t* idx;    // [T, k]; NULL: slot is the row (contiguous layout)
  const int32_t* slot;   // [T, k]
  const float* w;        // [T, k]
  int64_t T, top_k;
  const int32_t* num_valid;  // nullable device scalar: tokens >= *num_valid are not written
  uint16_t* out;             // bf16 [T, K]
};

// Row of route j of token t in expert_out, or -1 when the route is unrouted
// or out of range; its weight goes to *w.
__device__ __forceinline__ int64_t route_row(const ReduceParams& p, int64_t t, int64_t j,
                                             float* w) {
  const int32_t s = p.slot[t * p.top_k + j];
  *w = p.w[t * p.top_k + j];
  if (p.idx != nullptr) {  // batched: (expert, slot)
    const int64_t e = p.idx[t * p.top_k + j];
    return (e >= 0 && s >= 0 && e < p.E && s < p.M_max) ? e * p.M_max + s : -1;
  }
  return (s >= 0 && s < p.E * p.M_max) ? (int64_t)s : -1;  // contiguous: the slot is the row
}

__global__ void __launch_bounds__(256) topk_reduce_kernel(ReduceParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t gwarp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  // tasks index (token, 256-column chunk) pairs; the host keeps T * chunks < 2^31
  const uint32_t chunks = (uint32_t)((p.K + 255) / 256);
  pdl_wait();
  pdl_launch_dependents();
  // the device-side token bound (a captured graph can run smaller batches)
  int64_t T = p.T;
  if (p.num_valid != nullptr) {
    const int64_t nv = *p.num_valid;
    T = nv < 0 ? 0 : (nv < T ? nv : T);
  }
  const uint32_t tasks = (uint32_t)(T * chunks);
  for (uint32_t task = (uint32_t)gwarp; task < tasks; task += (uint32_t)nwarps) {
    const uint32_t tq = task / chunks;
    const int64_t t = tq;
    const int64_t c0 = (int64_t)(task - tq * chunks) * 256 + lane * 8;
    const bool active = c0 < p.K;
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    // Lane j < min(top_k, 32) resolves route j's row and weight once; the
    // rows are then read in groups of 8 with all loads in flight before the
    // sums, which stay in ascending j.  Routes past 32 resolve directly.
    int64_t my_row = -1;
    float my_w = 0.0f;
    if (lane < p.top_k) my_row = route_row(p, t, lane, &my_w);
    for (int64_t j0 = 0; j0 < p.top_k; j0 += 8) {
      uint4 v[8];
      float wt[8];
      bool use[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int64_t j = j0 + i;  // warp-uniform
        int64_t row = -1;
        wt[i] = 0.0f;
        if (j < 32) {
          row = __shfl_sync(0xFFFFFFFFu, my_row, (int)j);
          wt[i] = __shfl_sync(0xFFFFFFFFu, my_w, (int)j);
        } else if (j < p.top_k) {
          row = route_row(p, t, j, &wt[i]);
        }
        use[i] = j < p.top_k && row >= 0;
        v[i] = (use[i] && active) ? ld_stream_v4(p.expert_out + row * p.K + c0)
                                  : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (!use[i]) continue;
        const uint32_t u[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          acc[2 * q] = fmaf(wt[i], bf16_bits_to_f32(u[q] & 0xFFFFu), acc[2 * q]);
          acc[2 * q + 1] = fmaf(wt[i], bf16_bits_to_f32(u[q] >> 16), acc[2 * q + 1]);
        }
      }
    }
    if (active) {
      uint4 o;
      o.x = f32_to_bf16_bits(acc[0]) | (f32_to_bf16_bits(acc[1]) << 16);
      o.y = f32_to_bf16_bits(acc[2]) | (f32_to_bf16_bits(acc[3]) << 16);
      o.z = f32_to_bf16_bits(acc[4]) | (f32_to_bf16_bits(acc[5]) << 16);
      o.w = f32_to_bf16_bits(acc[6]) | (f32_to_bf16_bits(acc[7]) << 16);
      st_v4(p.out + t * p.K + c0, o);
    }
  }
}

}  // namespace moe

namespace moe_host {

moe_status_t launch_topk_reduce(const void* expert_out, int64_t E, int64_t M_max, int64_t K,
                                const int64_t* idx, const int32_t* slot, const float* w,
                                int64_t T, int64_t top_k, const int32_t* num_valid, void* out,
                                cudaStream_t s) {
  moe::ReduceParams p{static_cast<const uint16_t*>(expert_out), E, M_max, K, idx, slot, w, T,
                      top_k, num_valid, static_cast<uint16_t*>(out)};
  const int64_t tasks = T * ((K + 255) / 256);
  int64_t blocks = (tasks * 32 + 255) / 256;
  const int64_t cap =
      (int64_t)num_sms() * resident_blocks(reinterpret_cast<const void*>(moe::topk_reduce_kernel), 256);
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  cudaError_t e = launch_pdl(moe::topk_reduce_kernel, dim3((unsigned)blocks), dim3(256), 0, s, p);
  if (e != cudaSuccess) return set_error(MOE_ERR_CUDA, "reduce launch: %s", cudaGetErrorString(e));
  return MOE_OK;
}

}  // namespace moe_host
