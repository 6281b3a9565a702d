// Input staging: bf16 -> fp8 e4m3 with 1x128 UE8M0 (or fp32) group scales,
// top-k repack with EPLB replica mapping, and the dispatch into the batched
// [E, M_max, K] layout.
//
// Follows prepare_megamoe_inputs / _quantize_fp8_groups / _pack_bytes /
// _store_topk / _eplb_kernel_args ("vllm.model_executor.layers.fused_moe.
// prepare_megamoe") and the BatchedExperts activation format of
// BatchedHummingGroupedExperts ("...fused_moe.experts.fused_humming_moe").
//
// Kernels
//   small_dispatch_kernel : a batch of at most 1024 routes with dispatch, in
//                  one launch: every block ranks all routes in shared memory,
//                  then quantises its tasks and scatters them.
//   route_kernel : one thread per route (t, j), 1024 routes per block.  Repack
//                  + EPLB + per-block expert histogram + the stable rank of the
//                  route among the block's routes to the same expert.  The last
//                  block to finish turns the histograms into per-block
//                  exclusive offsets (column scan over blocks) and writes
//                  expert_num_tokens.
//   quant_ring_kernel : batches of 1024 tokens or more: rows stream through
//                  shared-memory buffers filled by bulk copies, one per row
//                  warp, with two routing warps repacking alongside.
//   quant_kernel : shorter batches: one warp per (token, 4 groups = 512
//                  elements): two 16-byte loads per lane, each covering 512
//                  contiguous bytes per warp, warp-shuffle amax over the 16
//                  lanes of a group, packed fp8 stores, one packed exponent
//                  word per task; optionally the same bytes are stored into
//                  each routed slot of x_b.
//   nvfp4_ring_kernel / nvfp4_kernel : the NVFP4 token staging, in the same
//                  two forms.
//                  Without dispatch the repack is folded into the quantiser.
#include <cstdio>
#include <type_traits>

#include <cuda_fp16.h>

#include "common.cuh"

namespace moe {

struct StageParams {
  int64_t T, K, top_k, G, W;  // W = ceil(G/4) packed words per row
  const uint16_t* hidden;
  int64_t hs0;
  const void* ids;
  int64_t is0, is1;
  const void* wts;
  int64_t ws0, ws1;
  const uint8_t* pad;
  int64_t ps0;
  uint8_t* x;
  int64_t xs0;
  void* x_sf;
  int64_t sfs0, sfs1;
  uint8_t* shared_sf;  // shared-expert scale pages (nullable)
  int64_t ss0, ss1, sbm, sbm_aligned;
  int sf_word;         // pages take a token's 4 exponent bytes as one 32-bit store
  int64_t* ids_out;
  int64_t ios0, ios1;
  float* w_out;
  int64_t wos0, wos1;
  const int32_t* l2p;
  int64_t num_logical, map_stride;
  const int32_t* rep_count;
  int32_t* load;
  int64_t num_physical;
  const uint8_t* record;
  const int32_t* num_unpadded;
  // dispatch
  int64_t E, M_max;
  uint8_t* x_b;
  int32_t* sf_b;        // packed UE8M0 words [rows, W], or fp32 [rows, G] (FP32 mode)
  int32_t* expert_num_tokens;
  int32_t* route_slot;
  int32_t* offsets;     // contiguous layout: [E+1] first row of each expert (nullable)
  int32_t* hist;        // [B, E] -> exclusive offsets after the scan
  int32_t* local_rank;  // [T*k]
  uint32_t* done;       // block completion counter (zeroed by the host)
  int64_t num_route_blocks;
  uint32_t* status;
};

// Repack one route (t, j): int64 id (-1 for padding), fp32 weight, EPLB map and
// load record.  Returns the id written.  With WRITE false only the id is
// worked out: nothing is stored, counted or flagged.
template <typename IdT, typename WT, bool WRITE = true>
__device__ __forceinline__ int64_t repack_route(const StageParams& p, int64_t t, int64_t j,
                                                bool record_on, int64_t unpadded,
                                                int* smem_load = nullptr) {
  bool is_pad = p.pad ? (p.pad[t * p.ps0] != 0) : false;
  int64_t id = (int64_t)(reinterpret_cast<const IdT*>(p.ids)[t * p.is0 + j * p.is1]);
  float w;
  if constexpr (sizeof(WT) == 4) {
    w = reinterpret_cast<const float*>(p.wts)[t * p.ws0 + j * p.ws1];
  } else {
    w = bf16_bits_to_f32(reinterpret_cast<const uint16_t*>(p.wts)[t * p.ws0 + j * p.ws1]);
  }
  if (is_pad) {
    id = -1;
    w = 0.0f;
  }
  if (p.l2p != nullptr && id >= 0) {
    if (id >= p.num_logical) {
      if (WRITE) set_status(p.status, MOE_DEV_BAD_EXPERT);
      id = -1;
    } else {
      int32_t reps = p.rep_count[id];
      if (reps < 1) {
        if (WRITE) set_status(p.status, MOE_DEV_BAD_EXPERT);
        id = -1;
      } else {
        int64_t phys = p.l2p[id * p.map_stride + (t % reps)];
        if (phys < 0 || (p.load != nullptr && phys >= p.num_physical)) {
          if (WRITE) set_status(p.status, MOE_DEV_BAD_EXPERT);
          id = -1;
        } else {
          id = phys;
          if (WRITE && p.load != nullptr && record_on && t < unpadded) {
            if (smem_load != nullptr)
              atomicAdd(&smem_load[phys], 1);
            else
              atomicAdd(&p.load[phys], 1);
          }
        }
      }
    }
  }
  if constexpr (WRITE) {
    p.ids_out[t * p.ios0 + j * p.ios1] = id;
    p.w_out[t * p.wos0 + j * p.wos1] = w;
  }
  return id;
}

// The repack of routes r, r + stride, ... below R, four routes per thread at
// a time: the padding flag, id and weight loads of the four are issued
// together, then their replica counts, then their physical ids, so that each
// dependent load of the EPLB map is paid once per four routes instead of once
// per route.  Same results as repack_route on each route.
template <typename IdT, typename WT>
__device__ __forceinline__ void repack_strided(const StageParams& p, int64_t r, int64_t stride,
                                               int64_t R, bool record_on, int64_t unpadded,
                                               int* smem_load) {
  constexpr int U = 4;
  for (; r < R; r += stride * U) {
    int64_t id[U], t[U], j[U];
    float w[U];
    bool act[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t ru = r + u * stride;
      act[u] = ru < R;
      t[u] = act[u] ? ru / p.top_k : 0;
      j[u] = act[u] ? ru - t[u] * p.top_k : 0;
      id[u] = -1;
      w[u] = 0.0f;
      if (act[u]) {
        const bool is_pad = p.pad ? (p.pad[t[u] * p.ps0] != 0) : false;
        id[u] = (int64_t)(reinterpret_cast<const IdT*>(p.ids)[t[u] * p.is0 + j[u] * p.is1]);
        if constexpr (sizeof(WT) == 4) {
          w[u] = reinterpret_cast<const float*>(p.wts)[t[u] * p.ws0 + j[u] * p.ws1];
        } else {
          w[u] = bf16_bits_to_f32(
              reinterpret_cast<const uint16_t*>(p.wts)[t[u] * p.ws0 + j[u] * p.ws1]);
        }
        if (is_pad) {
          id[u] = -1;
          w[u] = 0.0f;
        }
      }
    }
    if (p.l2p != nullptr) {
      int32_t reps[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        reps[u] = 0;
        if (act[u] && id[u] >= 0) {
          if (id[u] >= p.num_logical) {
            set_status(p.status, MOE_DEV_BAD_EXPERT);
            id[u] = -1;
          } else {
            reps[u] = p.rep_count[id[u]];
          }
        }
      }
      int64_t phys[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        phys[u] = -1;
        if (act[u] && id[u] >= 0 && reps[u] >= 1)
          phys[u] = p.l2p[id[u] * p.map_stride + (t[u] % reps[u])];
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (!(act[u] && id[u] >= 0)) continue;
        if (reps[u] < 1 || phys[u] < 0 || (p.load != nullptr && phys[u] >= p.num_physical)) {
          set_status(p.status, MOE_DEV_BAD_EXPERT);
          id[u] = -1;
        } else {
          id[u] = phys[u];
          if (p.load != nullptr && record_on && t[u] < unpadded) {
            if (smem_load != nullptr)
              atomicAdd(&smem_load[phys[u]], 1);
            else
              atomicAdd(&p.load[phys[u]], 1);
          }
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (!act[u]) continue;
      p.ids_out[t[u] * p.ios0 + j[u] * p.ios1] = id[u];
      p.w_out[t[u] * p.wos0 + j[u] * p.wos1] = w[u];
    }
  }
}

__device__ __forceinline__ void record_flags(const StageParams& p, bool& record_on,
                                             int64_t& unpadded) {
  record_on = p.record != nullptr && (*p.record != 0);
  unpadded = p.num_unpadded != nullptr ? (int64_t)(*p.num_unpadded) : p.T;
}

// ---------------------------------------------------------------------------
// route_kernel: repack + EPLB + stable within-block ranks + histogram scan.
// blockDim = 1024; dynamic smem = 32 * E uint16 warp counts.
// ---------------------------------------------------------------------------
template <typename IdT, typename WT>
__global__ void __launch_bounds__(1024) route_kernel(StageParams p) {
  extern __shared__ uint16_t warp_cnt[];  // [32][E]
  __shared__ int s_last;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t R = p.T * p.top_k;
  const int64_t r = (int64_t)blockIdx.x * 1024 + tid;
  const int E = (int)p.E;

  for (int i = tid; i < 32 * E; i += 1024) warp_cnt[i] = 0;
  pdl_wait();
  pdl_launch_dependents();

  bool record_on;
  int64_t unpadded;
  record_flags(p, record_on, unpadded);

  int e = -1;
  if (r < R) {
    int64_t t = r / p.top_k, j = r % p.top_k;
    int64_t id = repack_route<IdT, WT>(p, t, j, record_on, unpadded);
    if (id >= E) {
      set_status(p.status, MOE_DEV_BAD_EXPERT);
      id = -1;
    }
    e = (int)id;
  }
  __syncthreads();  // warp_cnt zeroed

  // Stable rank among this warp's routes to the same expert.
  const uint32_t same = __match_any_sync(0xFFFFFFFFu, e);
  const int rank_in_warp = __popc(same & lanemask_lt());
  if (e >= 0 && rank_in_warp == 0) warp_cnt[warp * E + e] = (uint16_t)__popc(same);
  __syncthreads();
  if (e >= 0) {
    int base = 0;
    for (int w = 0; w < warp; ++w) base += warp_cnt[w * E + e];
    p.local_rank[r] = base + rank_in_warp;
  }
  // Block histogram row.
  for (int ex = tid; ex < E; ex += 1024) {
    int tot = 0;
#pragma unroll 8
    for (int w = 0; w < 32; ++w) tot += warp_cnt[w * E + ex];
    p.hist[(int64_t)blockIdx.x * E + ex] = tot;
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = (atomicAdd(p.done, 1u) == gridDim.x - 1) ? 1 : 0;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // Last block: column-wise exclusive scan of hist over blocks (E <= 1024,
  // so each thread owns at most one expert).
  const int64_t B = p.num_route_blocks;
  int run = 0;
  if (tid < E) {
    for (int64_t b = 0; b < B; ++b) {
      int v = __ldcg(&p.hist[b * E + tid]);
      p.hist[b * E + tid] = run;
      run += v;
    }
  }
  if (p.offsets == nullptr) {
    if (tid < E) {
      if (run > p.M_max) set_status(p.status, MOE_DEV_CAPACITY);
      p.expert_num_tokens[tid] = (int32_t)min((int64_t)run, p.M_max);
    }
  } else {
    // Contiguous layout: exclusive scan of the per-expert totals over the
    // experts gives each expert's first row; it is added to every block's
    // offset so that a route's slot becomes its row.
    __shared__ int s_warp_tot[32];
    int incl = run;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
      if (lane >= off) incl += o;
    }
    if (lane == 31) s_warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int v = s_warp_tot[lane];
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xFFFFFFFFu, v, off);
        if (lane >= off) v += o;
      }
      s_warp_tot[lane] = v;  // inclusive over warps
    }
    __syncthreads();
    const int base = incl - run + (warp > 0 ? s_warp_tot[warp - 1] : 0);
    if (tid < E) {
      for (int64_t b = 0; b < B; ++b) p.hist[b * E + tid] += base;
      p.offsets[tid] = base;
      p.expert_num_tokens[tid] = run;
    }
    if (tid == E - 1) p.offsets[E] = base + run;
  }
  if (tid == 0) *p.done = 0u;
}

// ---------------------------------------------------------------------------
// quant_kernel: one warp per (token t, word w) task = groups 4w .. 4w+3
// (512 elements).  Each of the two 16-byte loads of the warp covers 512
// contiguous bytes: load A holds groups 4w (lanes 0-15) and 4w+1 (lanes
// 16-31), load B groups 4w+2 and 4w+3.  A group's amax is reduced over its 16
// lanes; every lane stores its 8 fp8 codes of each load (256 contiguous bytes
// per warp store).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float amax8(uint4 v, float f[8]) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = bf16_bits_to_f32(u[i] & 0xFFFFu);
    f[2 * i + 1] = bf16_bits_to_f32(u[i] >> 16);
    m = fmaxf(m, fmaxf(fabsf(f[2 * i]), fabsf(f[2 * i + 1])));
  }
  // reduce over the 16 lanes that share the group
  m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 8));
  m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 4));
  m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
  m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
  return m;
}

template <int SF_MODE>
__device__ __forceinline__ uint2 quant8(const float f[8], float amax, uint32_t& code) {
  float inv;
  if constexpr (SF_MODE == MOE_SF_UE8M0_PACKED) {
    code = ue8m0_exponent(amax);
    inv = ue8m0_inverse(code);
  } else {
    const float s = __fdiv_rn(fmaxf(amax, 1.0e-4f), 448.0f);
    code = __float_as_uint(s);
    inv = __frcp_rn(s);
  }
  uint2 q;
  q.x = pack4_e4m3(__fmul_rn(f[0], inv), __fmul_rn(f[1], inv), __fmul_rn(f[2], inv),
                   __fmul_rn(f[3], inv));
  q.y = pack4_e4m3(__fmul_rn(f[4], inv), __fmul_rn(f[5], inv), __fmul_rn(f[6], inv),
                   __fmul_rn(f[7], inv));
  return q;
}

__device__ __forceinline__ void st_v2(void* p, uint2 v) {
  asm volatile("st.global.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}

// One task after its two loads have landed.  With SMALL the destination row
// of every route comes ready-made from srows (-1: not dispatched) and
// route_slot is written elsewhere.
template <int SF_MODE, bool DISPATCH, bool SHARED, bool SMALL = false>
__device__ __forceinline__ void quant_task(const StageParams& p, int64_t t, int64_t w, uint4 vA,
                                           uint4 vB, int lane, const int32_t* srows = nullptr) {
  const int half = lane >> 4;
  const int64_t gA = 4 * w + half, gB = 4 * w + 2 + half;
  const bool actA = gA < p.G, actB = gB < p.G;
  const int64_t e0 = 4 * w * kGroup;
  const int64_t offA = e0 + lane * 8, offB = e0 + 256 + lane * 8;
  if constexpr (SF_MODE == MOE_SF_NONE) {
    uint16_t* dst = reinterpret_cast<uint16_t*>(p.x) + t * p.xs0;
    if (actA) st_v4(dst + offA, vA);
    if (actB) st_v4(dst + offB, vB);
  } else {
    float fA[8], fB[8];
    const float mA = amax8(vA, fA);
    const float mB = amax8(vB, fB);
    uint32_t cA, cB;
    const uint2 qA = quant8<SF_MODE>(fA, mA, cA);
    const uint2 qB = quant8<SF_MODE>(fB, mB, cB);
    uint8_t* xrow = p.x + t * p.xs0;
    if (actA) st_v2(xrow + offA, qA);
    if (actB) st_v2(xrow + offB, qB);

    uint32_t word = 0;
    if constexpr (SF_MODE == MOE_SF_UE8M0_PACKED) {
      const uint32_t a = actA ? cA : 0u, b = actB ? cB : 0u;
      const uint32_t e0w = __shfl_sync(0xFFFFFFFFu, a, 0);
      const uint32_t e1w = __shfl_sync(0xFFFFFFFFu, a, 16);
      const uint32_t e2w = __shfl_sync(0xFFFFFFFFu, b, 0);
      const uint32_t e3w = __shfl_sync(0xFFFFFFFFu, b, 16);
      word = e0w | (e1w << 8) | (e2w << 16) | (e3w << 24);
      if (lane == 0) reinterpret_cast<uint32_t*>(p.x_sf)[t * p.sfs0 + w * p.sfs1] = word;
      if constexpr (SHARED) {
        // shared-expert pages: each 128-row page holds its four 32-token
        // quarters interleaved row by row.  A page row keeps the token's
        // exponent bytes in group order, so the packed word goes in one
        // 32-bit store when the pages allow it (else byte by byte).
        const int64_t m = t % p.sbm;
        const int64_t row = (t / p.sbm) * p.sbm_aligned + (m / 128) * 128 + (m % 32) * 4 +
                            (m % 128) / 32;
        if (p.sf_word && 4 * w + 3 < p.G) {
          if (lane == 0) *reinterpret_cast<uint32_t*>(p.shared_sf + row * p.ss0 + 4 * w) = word;
        } else if (lane < 4 && 4 * w + lane < p.G) {
          p.shared_sf[row * p.ss0 + (4 * w + lane) * p.ss1] = (uint8_t)(word >> (8 * lane));
        }
      }
    } else {
      if ((lane & 15) == 0) {
        float* sf = reinterpret_cast<float*>(p.x_sf) + t * p.sfs0;
        if (actA) sf[gA * p.sfs1] = __uint_as_float(cA);
        if (actB) sf[gB * p.sfs1] = __uint_as_float(cB);
      }
    }

    if constexpr (DISPATCH) {
      const int64_t K = p.K;
      // Lane j works out route j's destination row (three dependent loads),
      // so the top_k chains run side by side; the rows are then broadcast.
      int64_t my_slot = -1, my_row = -1;
      if (SMALL && lane < p.top_k) {
        my_row = srows[t * p.top_k + lane];
      } else if (!SMALL && lane < p.top_k) {
        const int64_t r = t * p.top_k + lane;
        const int64_t e = p.ids_out[t * p.ios0 + lane * p.ios1];
        if (e >= 0 && e < p.E) {
          // contiguous layout: the scanned offsets already include the
          // expert's first row, so the slot is the row
          my_slot = (int64_t)__ldcg(&p.hist[(r >> 10) * p.E + e]) + p.local_rank[r];
          if (p.offsets != nullptr) {
            my_row = my_slot;
          } else if (my_slot < p.M_max) {
            my_row = e * p.M_max + my_slot;
          } else {
            my_slot = -1;
          }
        }
        if (w == 0) p.route_slot[r] = (int32_t)my_slot;
      }
      for (int64_t j = 0; j < p.top_k; ++j) {
        const int64_t row = __shfl_sync(0xFFFFFFFFu, my_row, (int)j);
        if (row >= 0) {
          uint8_t* brow = p.x_b + row * K;
          if (actA) st_v2(brow + offA, qA);
          if (actB) st_v2(brow + offB, qB);
          if constexpr (SF_MODE == MOE_SF_UE8M0_PACKED) {
            if (lane == 0) p.sf_b[row * p.W + w] = (int32_t)word;
          } else {  // fp32 scales [rows, G]
            if ((lane & 15) == 0) {
              float* sfb = reinterpret_cast<float*>(p.sf_b) + row * p.G;
              if (actA) sfb[gA] = __uint_as_float(cA);
              if (actB) sfb[gB] = __uint_as_float(cB);
            }
          }
        }
      }
    }
  }
}

// Shared-memory load histogram of the repack (physical experts) and the number
// of blocks that share the recorded routes.
constexpr int kLoadBins = 2048;
constexpr int kLoadBlocks = 24;

// Each warp keeps the loads of QUANT_BATCH tasks (4 KB) in flight, and issues
// the loads of its next batch before it quantises the current one.
constexpr int QUANT_BATCH = 4;

struct TaskBatch {
  uint4 vA[QUANT_BATCH], vB[QUANT_BATCH];
  uint32_t t[QUANT_BATCH], w[QUANT_BATCH];
};

__device__ __forceinline__ void load_batch(const StageParams& p, TaskBatch& b, uint32_t base,
                                           uint32_t nw, uint32_t tasks, uint32_t Wd, int lane) {
  const int half = lane >> 4;
#pragma unroll
  for (int i = 0; i < QUANT_BATCH; ++i) {
    const uint32_t task = base + i * nw;
    b.t[i] = task / Wd;
    b.w[i] = task - b.t[i] * Wd;
    b.vA[i] = make_uint4(0, 0, 0, 0);
    b.vB[i] = b.vA[i];
    if (task < tasks) {
      const uint16_t* src = p.hidden + (int64_t)b.t[i] * p.hs0 + 4 * b.w[i] * kGroup + lane * 8;
      if (4 * b.w[i] + half < p.G) b.vA[i] = ld_stream_v4(src);
      if (4 * b.w[i] + 2 + half < p.G) b.vB[i] = ld_stream_v4(src + 256);
    }
  }
}

// The task loop of one warp: tasks base, base + nw, ... below `tasks`, with
// the first batch (cur) already loaded; each batch's successor is loaded
// before the batch is quantised.
template <int SF_MODE, bool DISPATCH, bool SHARED, bool SMALL>
__device__ __forceinline__ void quant_loop(const StageParams& p, TaskBatch& cur, uint32_t base,
                                           uint32_t nw, uint32_t tasks, int lane,
                                           const int32_t* srows) {
  const uint32_t Wd = (uint32_t)p.W;
  const uint32_t step = QUANT_BATCH * nw;
  TaskBatch nxt;
  for (; base < tasks; base += step) {
    const bool more = base + step < tasks;
    if (more) load_batch(p, nxt, base + step, nw, tasks, Wd, lane);
#pragma unroll
    for (int i = 0; i < QUANT_BATCH; ++i) {
      if (base + i * nw < tasks)
        quant_task<SF_MODE, DISPATCH, SHARED, SMALL>(p, cur.t[i], cur.w[i], cur.vA[i],
                                                     cur.vB[i], lane, srows);
    }
    if (more) cur = nxt;
  }
}

// Repack of routes [r0, r1) with the EPLB load counted in a shared-memory
// histogram that is added to the global counters once per non-zero bin.
// Per-route global atomics would land on the few L2 lines that hold the
// counters and serialise there.
template <typename IdT, typename WT>
__device__ __forceinline__ void repack_recorded(const StageParams& p, int64_t r0, int64_t r1,
                                                int64_t unpadded, int* s_load) {
  for (int i = threadIdx.x; i < p.num_physical; i += blockDim.x) s_load[i] = 0;
  __syncthreads();
  repack_strided<IdT, WT>(p, r0 + threadIdx.x, blockDim.x, r1, true, unpadded, s_load);
  __syncthreads();
  for (int i = threadIdx.x; i < p.num_physical; i += blockDim.x)
    if (s_load[i] != 0) atomicAdd(&p.load[i], s_load[i]);
}

template <int SF_MODE, bool REPACK, bool DISPATCH, typename IdT, typename WT, bool SHARED>
__global__ void __launch_bounds__(256) quant_kernel(StageParams p) {
  __shared__ int s_load[REPACK ? kLoadBins : 1];
  const int lane = threadIdx.x & 31;
  pdl_wait();
  pdl_launch_dependents();

  bool record_on = false;
  int64_t unpadded = p.T;
  if constexpr (REPACK) record_flags(p, record_on, unpadded);
  const int64_t R = p.T * p.top_k;
  // With load recording on, the repack runs in a few blocks of its own that
  // take contiguous route ranges; when the grid is large enough they are
  // set aside from the streaming so that their dependent-load chains overlap
  // it instead of trailing it.
  const bool recorded = REPACK && record_on && p.load != nullptr && p.num_physical <= kLoadBins;
  const int64_t nrep = recorded ? min((int64_t)gridDim.x, (int64_t)kLoadBlocks) : 0;
  const bool set_aside = recorded && gridDim.x >= 4 * kLoadBlocks;
  if constexpr (REPACK) {
    if (set_aside && blockIdx.x < nrep) {
      const int64_t per = (R + nrep - 1) / nrep;
      repack_recorded<IdT, WT>(p, blockIdx.x * per, min(R, (blockIdx.x + 1) * per), unpadded,
                               s_load);
      return;
    }
  }
  const int64_t sblock = set_aside ? blockIdx.x - nrep : blockIdx.x;
  const int64_t sgrid = set_aside ? gridDim.x - nrep : gridDim.x;
  const int64_t gwarp = (sblock * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (sgrid * blockDim.x) >> 5;

  // tasks index (token, word) pairs; the host guarantees T * W < 2^31
  const uint32_t tasks = (uint32_t)(p.T * p.W);
  TaskBatch cur;
  if ((uint32_t)gwarp < tasks) load_batch(p, cur, (uint32_t)gwarp, (uint32_t)nwarps, tasks,
                                          (uint32_t)p.W, lane);
  quant_loop<SF_MODE, DISPATCH, SHARED, false>(p, cur, (uint32_t)gwarp, (uint32_t)nwarps, tasks,
                                               lane, nullptr);

  // Without recording (or on a small grid) the top-k repack (dependent
  // loads, no bandwidth) goes last so that its latency overlaps the other
  // warps' streaming.
  if constexpr (REPACK) {
    if (recorded) {
      if (!set_aside && blockIdx.x < nrep) {
        const int64_t per = (R + nrep - 1) / nrep;
        repack_recorded<IdT, WT>(p, blockIdx.x * per, min(R, (blockIdx.x + 1) * per), unpadded,
                                 s_load);
      }
    } else {
      repack_strided<IdT, WT>(p, (int64_t)blockIdx.x * blockDim.x + threadIdx.x,
                              (int64_t)gridDim.x * blockDim.x, R, record_on, unpadded, nullptr);
    }
  }
}


// ---------------------------------------------------------------------------
// small_dispatch_kernel: the staging and dispatch of a batch of at most
// kSmallRoutes routes in one launch, with no workspace and no host memset.
// Every block maps all routes to their physical expert and ranks them in
// route order (at most four 256-route passes over shared memory), so that no
// block waits for another; block 0 alone stores the repacked ids and weights,
// the EPLB load record, route_slot and the per-expert counts (and the
// contiguous layout's first rows).  The first batch of hidden-state loads is
// issued before the routing, so the two overlap; the blocks then quantise
// their tasks and store each into its routed rows as quant_kernel does.
// Dynamic smem: E ints (running counts, then first rows) + 8 * E uint16
// (per-warp counts of one pass).
// ---------------------------------------------------------------------------
constexpr int kSmallRoutes = 1024;

template <int SF_MODE, typename IdT, typename WT, bool SHARED>
__global__ void __launch_bounds__(256) small_dispatch_kernel(StageParams p) {
  extern __shared__ int32_t s_dyn[];
  __shared__ int32_t s_row[kSmallRoutes];  // rank, then destination row (-1: none)
  __shared__ int16_t s_e[kSmallRoutes];    // physical expert (-1: unrouted)
  __shared__ int32_t s_wsum[8];
  const int E = (int)p.E;
  int32_t* s_run = s_dyn;
  uint16_t* s_cnt = reinterpret_cast<uint16_t*>(s_dyn + E);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int R = (int)(p.T * p.top_k);
  const bool lead = blockIdx.x == 0;
  for (int i = tid; i < 5 * E; i += 256) s_dyn[i] = 0;  // E + 8E/2 words
  pdl_wait();

  // the first batch of this warp's tasks is in flight during the routing
  const uint32_t tasks = (uint32_t)(p.T * p.W);
  const uint32_t gwarp = (uint32_t)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const uint32_t nwarps = (uint32_t)((gridDim.x * blockDim.x) >> 5);
  TaskBatch cur;
  if (gwarp < tasks) load_batch(p, cur, gwarp, nwarps, tasks, (uint32_t)p.W, lane);

  bool record_on;
  int64_t unpadded;
  record_flags(p, record_on, unpadded);
  for (int r = tid; r < R; r += 256) {
    const int64_t t = r / p.top_k, j = r - t * p.top_k;
    int64_t id = lead ? repack_route<IdT, WT, true>(p, t, j, record_on, unpadded)
                      : repack_route<IdT, WT, false>(p, t, j, record_on, unpadded);
    if (id >= E) {
      if (lead) set_status(p.status, MOE_DEV_BAD_EXPERT);
      id = -1;
    }
    s_e[r] = (int16_t)id;
  }
  __syncthreads();

  // Stable rank of each route among the routes to its expert: 256 routes per
  // pass in route order; within a pass, warps in order and lanes in order.
  for (int c = 0; c < R; c += 256) {
    const int r = c + tid;
    const int e = r < R ? s_e[r] : -1;
    const uint32_t same = __match_any_sync(0xFFFFFFFFu, e);
    const int rank_in_warp = __popc(same & lanemask_lt());
    if (e >= 0 && rank_in_warp == 0) s_cnt[warp * E + e] = (uint16_t)__popc(same);
    __syncthreads();
    if (e >= 0) {
      int base = s_run[e];
      for (int w = 0; w < warp; ++w) base += s_cnt[w * E + e];
      s_row[r] = base + rank_in_warp;
    }
    __syncthreads();
    for (int ex = tid; ex < E; ex += 256) {
      int tot = 0;
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        tot += s_cnt[w * E + ex];
        s_cnt[w * E + ex] = 0;
      }
      s_run[ex] += tot;
    }
    __syncthreads();
  }

  // s_run[e] = routes to expert e.  Ranks become destination rows.
  if (p.offsets == nullptr) {
    if (lead) {
      for (int ex = tid; ex < E; ex += 256) {
        const int n = s_run[ex];
        if (n > p.M_max) set_status(p.status, MOE_DEV_CAPACITY);
        p.expert_num_tokens[ex] = (int32_t)min((int64_t)n, p.M_max);
      }
    }
    for (int r = tid; r < R; r += 256) {
      const int e = s_e[r];
      const int slot = (e >= 0 && s_row[r] < p.M_max) ? s_row[r] : -1;
      if (lead) p.route_slot[r] = slot;
      s_row[r] = slot >= 0 ? (int32_t)(e * p.M_max + slot) : -1;
    }
  } else {
    // contiguous layout: each expert's first row is the exclusive scan of
    // the counts over the experts; thread i owns experts [i*per, i*per+per)
    const int per = (E + 255) / 256;
    const int e0 = tid * per;
    int loc = 0;
    for (int i = 0; i < per; ++i)
      if (e0 + i < E) loc += s_run[e0 + i];
    int incl = loc;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
      if (lane >= off) incl += o;
    }
    if (lane == 31) s_wsum[warp] = incl;
    __syncthreads();
    int wbase = 0;
    for (int w = 0; w < warp; ++w) wbase += s_wsum[w];
    int first = wbase + incl - loc;
    for (int i = 0; i < per; ++i) {
      if (e0 + i >= E) break;
      const int n = s_run[e0 + i];
      if (lead) {
        p.offsets[e0 + i] = first;
        p.expert_num_tokens[e0 + i] = n;
      }
      s_run[e0 + i] = first;
      first += n;
    }
    if (lead && tid == 255) p.offsets[E] = wbase + incl;
    __syncthreads();
    for (int r = tid; r < R; r += 256) {
      const int e = s_e[r];
      const int row = e >= 0 ? s_run[e] + s_row[r] : -1;
      if (lead) p.route_slot[r] = row;
      s_row[r] = row;
    }
  }
  __syncthreads();
  // The next kernel is let in only now: a GEMM block launched during the
  // routing would take an SM that the routing's blocks still need, and the
  // whole step runs 3-5 us longer that way.
  pdl_launch_dependents();
  quant_loop<SF_MODE, true, SHARED, true>(p, cur, gwarp, nwarps, tasks, lane, s_row);
}

// ---------------------------------------------------------------------------
// NVFP4 token staging: per-token fp32 scale amax/2688, E2M1 codes with one
// E4M3 scale per 16 values.  One warp per token; lane l owns the 16-value
// blocks l, l+32, ... (two 16-byte loads each), so a block's scale, its
// reciprocal and its codes stay in one lane with no shuffles.  Rows of up to
// 32*NBL blocks are held in registers between the amax pass and the
// quantisation pass; longer rows (NBL = 0) are read twice, the second time
// from L2.
// ---------------------------------------------------------------------------
struct Nvfp4Params {
  int64_t T, K;
  const uint16_t* hidden;
  int64_t hs0;
  uint8_t* x;
  int64_t xs0;
  uint32_t* x_sf;
  int64_t sfs0;
  float* x_scales;
  uint16_t* shared_x;   // bf16 copy (MOE_SHARED_BF16)
  uint8_t* shared_q;    // fp8 MXFP8 shared input (MOE_SHARED_FP8)
  int64_t shs0;         // row stride of either, in its elements
  uint8_t* shared_sf;   // fp8 shared input: exponent bytes of the shared-expert pages
  int64_t ss0, ss1, sbm, sbm_aligned;
  const float* w2gs;
  float* l2_alpha;
  int64_t n_local;
  float l2s;
};

// E4M3 code -> fp32 (exact).
__device__ __forceinline__ float e4m3_to_f32(uint32_t code) {
  uint32_t h2;
  asm("{ .reg .b16 c; cvt.u16.u32 c, %1; cvt.rn.f16x2.e4m3x2 %0, c; }" : "=r"(h2) : "r"(code));
  return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}

// Eight fp32 -> eight E2M1 codes (round to nearest even, saturating to +-6),
// value 2i in the low nibble of byte i.
__device__ __forceinline__ uint32_t e2m1x8(const float* f) {
  uint32_t r;
  asm("{ .reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3}; }"
      : "=r"(r)
      : "f"(f[0]), "f"(f[1]), "f"(f[2]), "f"(f[3]), "f"(f[4]), "f"(f[5]), "f"(f[6]),
        "f"(f[7]));
  return r;
}

// Packed bf16x2 whose halves have magnitudes max(|a|, |b|) (the signs are
// the xor of the inputs' and are ignored; a NaN half yields the other one).
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Magnitude max over the 16 bf16 values of one block, as packed bf16x2.
__device__ __forceinline__ uint32_t block_absmax2(uint4 a, uint4 b) {
  return absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(a.x, a.y), absmax_bf16x2(a.z, a.w)),
                       absmax_bf16x2(absmax_bf16x2(b.x, b.y), absmax_bf16x2(b.z, b.w)));
}

__device__ __forceinline__ float absmax2_to_f32(uint32_t m) {
  return fmaxf(__uint_as_float((m & 0x7FFFu) << 16), __uint_as_float(m & 0x7FFF0000u));
}

// q = x / 6 without the divide's slow path: q0 = x * RN(1/6), the exact
// remainder r = x - 6 q0 by FMA, then one correction q0 + r * RN(1/6)
// (Markstein's correction step).  Over all 2^32 fp32 inputs this equals the
// IEEE quotient except where both are below 2^-126, where E4M3 encodes
// either one as 0.
__device__ __forceinline__ float div6(float x) {
  const float zh = 0.16666667163372039794921875f;  // RN(1/6)
  const float q0 = __fmul_rn(x, zh);
  const float r = __fmaf_rn(-q0, 6.0f, x);
  const float q = __fmaf_rn(r, zh, q0);
  return isinf(x) ? x : q;
}

// Quantise block b of token t (values in a, b2; magnitude max bm).  The
// block scale is E4M3(max|rn(x*inv)| / 6); rn is monotone, so that max is
// rn(max|x| * inv).  A block whose scale is 0 keeps zero codes.
__device__ __forceinline__ void nvfp4_block(const Nvfp4Params& q, const float* s_rcp, int64_t t,
                                            int64_t b, bool act, uint4 a, uint4 b2, uint32_t bm,
                                            float inv) {
  const float braw = absmax2_to_f32(bm);
  const float bmax = braw > 0.0f ? __fmul_rn(braw, inv) : 0.0f;
  const uint32_t sc = e4m3x2(div6(bmax), 0.0f) & 0xFFu;
  const float rs = s_rcp[sc & 0x7Fu];
  const uint32_t u[8] = {a.x, a.y, a.z, a.w, b2.x, b2.y, b2.z, b2.w};
  float f[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    f[2 * i] = __fmul_rn(__fmul_rn(bf16_bits_to_f32(u[i] & 0xFFFFu), inv), rs);
    f[2 * i + 1] = __fmul_rn(__fmul_rn(bf16_bits_to_f32(u[i] >> 16), inv), rs);
  }
  uint32_t c0 = e2m1x8(f), c1 = e2m1x8(f + 8);
  c0 = sc != 0 ? c0 : 0u;
  c1 = sc != 0 ? c1 : 0u;
  if (act) {
    uint32_t* xr = reinterpret_cast<uint32_t*>(q.x + t * q.xs0) + 2 * b;
    xr[0] = c0;
    xr[1] = c1;
    reinterpret_cast<uint8_t*>(q.x_sf + t * q.sfs0)[b] = (uint8_t)sc;  // byte b of the row
    if (q.shared_x != nullptr) {
      st_v4(q.shared_x + t * q.shs0 + b * 16, a);
      st_v4(q.shared_x + t * q.shs0 + b * 16 + 8, b2);
    }
  }
}

// The MXFP8 shared input of one 16-value block: the 1x128 group of block b
// is the 8 consecutive blocks 8g..8g+7, held by 8 consecutive lanes of the
// same register slot, so the group amax is a max over those 8 lanes of the
// blocks' magnitude maxima.  Codes and the exponent byte follow the fp8
// staging recipe (UE8M0 power of two, x * (1/qs) rounded to e4m3).  Every
// lane of the warp must call this (the groups of 8 lanes are either wholly
// inside the row or wholly past it).
__device__ __forceinline__ void shared_fp8_block(const Nvfp4Params& q, int64_t t, int64_t b,
                                                 bool act, uint4 a, uint4 b2, uint32_t bm) {
  float gm = absmax2_to_f32(bm);
  gm = fmaxf(gm, __shfl_xor_sync(0xFFFFFFFFu, gm, 1));
  gm = fmaxf(gm, __shfl_xor_sync(0xFFFFFFFFu, gm, 2));
  gm = fmaxf(gm, __shfl_xor_sync(0xFFFFFFFFu, gm, 4));
  const uint32_t code = ue8m0_exponent(gm);
  const float inv = ue8m0_inverse(code);
  if (act) {
    const uint32_t u[8] = {a.x, a.y, a.z, a.w, b2.x, b2.y, b2.z, b2.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      o[i] = pack4_e4m3(__fmul_rn(bf16_bits_to_f32(u[2 * i] & 0xFFFFu), inv),
                        __fmul_rn(bf16_bits_to_f32(u[2 * i] >> 16), inv),
                        __fmul_rn(bf16_bits_to_f32(u[2 * i + 1] & 0xFFFFu), inv),
                        __fmul_rn(bf16_bits_to_f32(u[2 * i + 1] >> 16), inv));
    st_v4(q.shared_q + t * q.shs0 + b * 16, make_uint4(o[0], o[1], o[2], o[3]));
    // one byte per group (gathering four groups into one 32-bit store
    // measured 4% slower here)
    if ((threadIdx.x & 7) == 0) {
      const int64_t m = t % q.sbm;
      const int64_t row = (t / q.sbm) * q.sbm_aligned + (m / 128) * 128 + (m % 32) * 4 +
                          (m % 128) / 32;
      q.shared_sf[row * q.ss0 + (b >> 3) * q.ss1] = (uint8_t)code;
    }
  }
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, off));
  return v;
}

template <typename IdT, typename WT, int NBL, bool SHARED_FP8>
__global__ void __launch_bounds__(128) nvfp4_kernel(Nvfp4Params q, StageParams p) {
  const int lane = threadIdx.x & 31;
  // RN(1 / dec(code)) for every E4M3 code of a non-negative scale (0x7F: NaN)
  __shared__ float s_rcp[128];
  for (int i = threadIdx.x; i < 128; i += blockDim.x) s_rcp[i] = __frcp_rn(e4m3_to_f32(i));
  __syncthreads();
  pdl_wait();
  pdl_launch_dependents();
  if (blockIdx.x == 0 && q.l2_alpha != nullptr)
    for (int64_t e = threadIdx.x; e < q.n_local; e += blockDim.x)
      q.l2_alpha[e] = __fmul_rn(q.w2gs[e], q.l2s);
  // routing: the same repack as the fp8 staging.  With load recording on and
  // a large grid, a few blocks are set aside for it from the start, so that
  // its dependent-load chains overlap the row streaming instead of trailing it.
  __shared__ int s_load[kLoadBins];
  bool record_on;
  int64_t unpadded;
  record_flags(p, record_on, unpadded);
  const int64_t R = p.T * p.top_k;
  const bool recorded = record_on && p.load != nullptr && p.num_physical <= kLoadBins;
  const int64_t nrep = recorded ? min((int64_t)gridDim.x, (int64_t)kLoadBlocks) : 0;
  const bool set_aside = recorded && gridDim.x >= 4 * kLoadBlocks;
  if (set_aside && blockIdx.x < nrep) {
    const int64_t per = (R + nrep - 1) / nrep;
    repack_recorded<IdT, WT>(p, blockIdx.x * per, min(R, (blockIdx.x + 1) * per), unpadded,
                             s_load);
    return;
  }
  const int64_t sblock = set_aside ? blockIdx.x - nrep : blockIdx.x;
  const int64_t sgrid = set_aside ? gridDim.x - nrep : gridDim.x;
  const int64_t swarp = (sblock * blockDim.x + threadIdx.x) >> 5;
  const int64_t snwarps = (sgrid * blockDim.x) >> 5;
  const int64_t nb = q.K / 16;  // a multiple of 8 (K % 128 == 0)
  for (int64_t t = swarp; t < q.T; t += snwarps) {
    const uint16_t* row = q.hidden + t * q.hs0;
    if constexpr (NBL > 0) {
      uint4 va[NBL], vb[NBL];
      uint32_t bm[NBL];
#pragma unroll
      for (int i = 0; i < NBL; ++i) {
        const int64_t b = lane + 32 * i;
        const bool in = b < nb;
        va[i] = in ? ld_stream_v4(row + b * 16) : make_uint4(0, 0, 0, 0);
        vb[i] = in ? ld_stream_v4(row + b * 16 + 8) : make_uint4(0, 0, 0, 0);
      }
      uint32_t m2 = 0;
#pragma unroll
      for (int i = 0; i < NBL; ++i) {
        bm[i] = block_absmax2(va[i], vb[i]);
        m2 = absmax_bf16x2(m2, bm[i]);
      }
      const float amax = warp_max(absmax2_to_f32(m2));
      const float xs = __fdiv_rn(amax, 2688.0f);
      if (lane == 0) q.x_scales[t] = xs;
      const float inv = amax > 0.0f ? __frcp_rn(xs) : 0.0f;
#pragma unroll
      for (int i = 0; i < NBL; ++i) {
        const int64_t b = lane + 32 * i;
        nvfp4_block(q, s_rcp, t, b, b < nb, va[i], vb[i], bm[i], inv);
        if constexpr (SHARED_FP8) shared_fp8_block(q, t, b, b < nb, va[i], vb[i], bm[i]);
      }
    } else {
      uint32_t m2 = 0;
      for (int64_t b = lane; b < nb; b += 32)
        m2 = absmax_bf16x2(m2, block_absmax2(ld_stream_v4(row + b * 16),
                                             ld_stream_v4(row + b * 16 + 8)));
      const float amax = warp_max(absmax2_to_f32(m2));
      const float xs = __fdiv_rn(amax, 2688.0f);
      if (lane == 0) q.x_scales[t] = xs;
      const float inv = amax > 0.0f ? __frcp_rn(xs) : 0.0f;
      // warp-uniform trip count: the shared input's group max is a shuffle
      for (int64_t b0 = 0; b0 < nb; b0 += 32) {
        const int64_t b = b0 + lane;
        const bool act = b < nb;
        const uint4 a = act ? ld_stream_v4(row + b * 16) : make_uint4(0, 0, 0, 0);
        const uint4 b2 = act ? ld_stream_v4(row + b * 16 + 8) : make_uint4(0, 0, 0, 0);
        const uint32_t bmx = block_absmax2(a, b2);
        nvfp4_block(q, s_rcp, t, b, act, a, b2, bmx, inv);
        if constexpr (SHARED_FP8) shared_fp8_block(q, t, b, act, a, b2, bmx);
      }
    }
  }
  if (recorded) {
    if (!set_aside && blockIdx.x < nrep) {
      const int64_t per = (R + nrep - 1) / nrep;
      repack_recorded<IdT, WT>(p, blockIdx.x * per, min(R, (blockIdx.x + 1) * per), unpadded,
                               s_load);
    }
  } else {
    repack_strided<IdT, WT>(p, (int64_t)blockIdx.x * blockDim.x + threadIdx.x,
                            (int64_t)gridDim.x * blockDim.x, R, record_on, unpadded, nullptr);
  }
}

// ---------------------------------------------------------------------------
// NVFP4 token staging for rows of up to 8192 values, streamed through shared
// memory.  One block per SM; each of its row warps owns a row buffer in
// shared memory, fills it with a 1-D bulk copy (cp.async.bulk, completion
// counted on the buffer's mbarrier) and quantises the landed row from shared
// memory, then refills the buffer with its next row.  As many row warps as
// row buffers fit in shared memory (up to RING_MAX_WARPS) keep that many rows
// in flight per SM, bounded by shared memory rather than by registers.  The
// last two warps do the top-k repack and EPLB map of the block's share of the
// routes at the same time.  Same per-row arithmetic as nvfp4_kernel
// (nvfp4_block, shared_fp8_block).  Measured on staging_stress with 4-14 row
// warps and one to three buffers each: more row warps win (12 or more).
// ---------------------------------------------------------------------------
constexpr int RING_MAX_WARPS = 14;
constexpr int RING_ROUTING_WARPS = 2;

__device__ __forceinline__ void bulk_row_load(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ bool ring_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for a row copy (2 s of globaltimer); false on expiry.
__device__ __forceinline__ bool ring_wait(uint32_t bar, uint32_t parity) {
  if (ring_try_wait(bar, parity)) return true;
  uint64_t t0;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  for (uint32_t it = 1;; ++it) {
    if (ring_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0u) {
      uint64_t t1;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t1));
      if (t1 - t0 > 2000000000ull) return false;
    }
  }
}

template <typename IdT, typename WT, int NBL, bool SHARED_FP8>
__global__ void __launch_bounds__((RING_MAX_WARPS + RING_ROUTING_WARPS) * 32, 1)
    nvfp4_ring_kernel(Nvfp4Params q, StageParams p) {
  extern __shared__ __align__(128) uint8_t ring_smem[];
  __shared__ float s_rcp[128];
  __shared__ __align__(8) uint64_t s_bar[RING_MAX_WARPS];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row_warps = (int)(blockDim.x >> 5) - RING_ROUTING_WARPS;
  const uint32_t rowbytes = (uint32_t)(q.K * 2);
  for (int i = threadIdx.x; i < 128; i += blockDim.x) s_rcp[i] = __frcp_rn(e4m3_to_f32(i));
  if (threadIdx.x == 0) {
    for (int i = 0; i < row_warps; ++i)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(
                       (uint32_t)__cvta_generic_to_shared(&s_bar[i]))
                   : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  pdl_wait();
  pdl_launch_dependents();
  if (blockIdx.x == 0 && q.l2_alpha != nullptr)
    for (int64_t e = threadIdx.x; e < q.n_local; e += blockDim.x)
      q.l2_alpha[e] = __fmul_rn(q.w2gs[e], q.l2s);
  bool record_on;
  int64_t unpadded;
  record_flags(p, record_on, unpadded);

  if (warp >= row_warps) {
    // ---------------------------------------------------------- routing
    const int rt = threadIdx.x - row_warps * 32;  // 0..63
    const int64_t R = p.T * p.top_k;
    const bool recorded = record_on && p.load != nullptr && p.num_physical <= kLoadBins;
    if (recorded) {
      // this block's contiguous share of the routes, counted in a shared
      // histogram (after the ring buffers) and added once per non-zero bin
      int* s_load = reinterpret_cast<int*>(ring_smem + row_warps * rowbytes);
      for (int i = rt; i < p.num_physical; i += 64) s_load[i] = 0;
      asm volatile("bar.sync 1, 64;" ::: "memory");
      const int64_t per = (R + gridDim.x - 1) / gridDim.x;
      const int64_t r0 = (int64_t)blockIdx.x * per, r1 = min(R, r0 + per);
      repack_strided<IdT, WT>(p, r0 + rt, 64, r1, true, unpadded, s_load);
      asm volatile("bar.sync 1, 64;" ::: "memory");
      for (int i = rt; i < p.num_physical; i += 64)
        if (s_load[i] != 0) atomicAdd(&p.load[i], s_load[i]);
    } else {
      repack_strided<IdT, WT>(p, (int64_t)blockIdx.x * 64 + rt, (int64_t)gridDim.x * 64, R,
                              record_on, unpadded, nullptr);
    }
    return;
  }

  // ---------------------------------------------------------- rows
  const int64_t stride = (int64_t)gridDim.x * row_warps;
  const int64_t t0 = (int64_t)blockIdx.x * row_warps + warp;
  const uint8_t* row = ring_smem + warp * rowbytes;
  const uint32_t row_s = (uint32_t)__cvta_generic_to_shared(row);
  const uint32_t bar = (uint32_t)__cvta_generic_to_shared(&s_bar[warp]);
  const int64_t nb = q.K / 16;
  if (t0 < q.T && lane == 0) bulk_row_load(row_s, q.hidden + t0 * q.hs0, rowbytes, bar);
  __syncwarp();
  uint32_t parity = 0;
  for (int64_t t = t0; t < q.T; t += stride) {
    if (!__all_sync(0xFFFFFFFFu, ring_wait(bar, parity))) {
      // a copy that has not landed in 2 s: report it, give it one more
      // bounded wait so that it is not in flight when the block exits, and
      // stop using the buffer
      set_status(p.status, MOE_DEV_TIMEOUT);
      ring_wait(bar, parity);
      break;
    }
    parity ^= 1u;
    uint32_t bm[NBL];
    uint32_t m2 = 0;
#pragma unroll
    for (int k = 0; k < NBL; ++k) {
      const int64_t b = lane + 32 * k;
      bm[k] = 0;
      if (b < nb) {
        const uint4 a = *reinterpret_cast<const uint4*>(row + b * 32);
        const uint4 c = *reinterpret_cast<const uint4*>(row + b * 32 + 16);
        bm[k] = block_absmax2(a, c);
        m2 = absmax_bf16x2(m2, bm[k]);
      }
    }
    const float amax = warp_max(absmax2_to_f32(m2));
    const float xs = __fdiv_rn(amax, 2688.0f);
    if (lane == 0) q.x_scales[t] = xs;
    const float inv = amax > 0.0f ? __frcp_rn(xs) : 0.0f;
#pragma unroll
    for (int k = 0; k < NBL; ++k) {
      const int64_t b = lane + 32 * k;
      const bool act = b < nb;
      const uint4 a = act ? *reinterpret_cast<const uint4*>(row + b * 32) : make_uint4(0, 0, 0, 0);
      const uint4 c =
          act ? *reinterpret_cast<const uint4*>(row + b * 32 + 16) : make_uint4(0, 0, 0, 0);
      nvfp4_block(q, s_rcp, t, b, act, a, c, bm[k], inv);
      if constexpr (SHARED_FP8) shared_fp8_block(q, t, b, act, a, c, bm[k]);
    }
    // the buffer is read: refill it with this warp's next row
    __syncwarp();
    if (t + stride < q.T) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      if (lane == 0) bulk_row_load(row_s, q.hidden + (t + stride) * q.hs0, rowbytes, bar);
      __syncwarp();
    }
  }
}

// ---------------------------------------------------------------------------
// The fp8 (1x128) staging of long batches, streamed through shared memory the
// same way as nvfp4_ring_kernel: one block per SM, each row warp fills its
// row buffer with a bulk copy and quantises the landed row task by task
// (quant_task: the same per-task arithmetic, stores, shared pages and
// dispatch scatter as quant_kernel).  With the repack folded in, the last two
// warps repack the block's share of the routes meanwhile.
// ---------------------------------------------------------------------------
template <int SF_MODE, bool REPACK, bool DISPATCH, typename IdT, typename WT, bool SHARED>
__global__ void __launch_bounds__((RING_MAX_WARPS + RING_ROUTING_WARPS) * 32, 1)
    quant_ring_kernel(StageParams p) {
  extern __shared__ __align__(128) uint8_t ring_smem[];
  __shared__ __align__(8) uint64_t s_bar[RING_MAX_WARPS];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row_warps = (int)(blockDim.x >> 5) - RING_ROUTING_WARPS;
  const uint32_t rowbytes = (uint32_t)(p.K * 2);
  if (threadIdx.x == 0) {
    for (int i = 0; i < row_warps; ++i)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(
                       (uint32_t)__cvta_generic_to_shared(&s_bar[i]))
                   : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  pdl_wait();
  pdl_launch_dependents();

  if (warp >= row_warps) {
    // ---------------------------------------------------------- routing
    if constexpr (REPACK) {
      bool record_on;
      int64_t unpadded;
      record_flags(p, record_on, unpadded);
      const int rt = threadIdx.x - row_warps * 32;  // 0..63
      const int64_t R = p.T * p.top_k;
      if (record_on && p.load != nullptr && p.num_physical <= kLoadBins) {
        int* s_load = reinterpret_cast<int*>(ring_smem + row_warps * rowbytes);
        for (int i = rt; i < p.num_physical; i += 64) s_load[i] = 0;
        asm volatile("bar.sync 1, 64;" ::: "memory");
        const int64_t per = (R + gridDim.x - 1) / gridDim.x;
        const int64_t r0 = (int64_t)blockIdx.x * per, r1 = min(R, r0 + per);
        repack_strided<IdT, WT>(p, r0 + rt, 64, r1, true, unpadded, s_load);
        asm volatile("bar.sync 1, 64;" ::: "memory");
        for (int i = rt; i < p.num_physical; i += 64)
          if (s_load[i] != 0) atomicAdd(&p.load[i], s_load[i]);
      } else {
        repack_strided<IdT, WT>(p, (int64_t)blockIdx.x * 64 + rt, (int64_t)gridDim.x * 64, R,
                                record_on, unpadded, nullptr);
      }
    }
    return;
  }

  // ---------------------------------------------------------- rows
  const int64_t stride = (int64_t)gridDim.x * row_warps;
  const int64_t t0 = (int64_t)blockIdx.x * row_warps + warp;
  const uint8_t* row = ring_smem + warp * rowbytes;
  const uint32_t row_s = (uint32_t)__cvta_generic_to_shared(row);
  const uint32_t bar = (uint32_t)__cvta_generic_to_shared(&s_bar[warp]);
  const int half = lane >> 4;
  if (t0 < p.T && lane == 0) bulk_row_load(row_s, p.hidden + t0 * p.hs0, rowbytes, bar);
  __syncwarp();
  uint32_t parity = 0;
  for (int64_t t = t0; t < p.T; t += stride) {
    if (!__all_sync(0xFFFFFFFFu, ring_wait(bar, parity))) {
      // a copy that has not landed in 2 s: report it, give it one more
      // bounded wait so that it is not in flight when the block exits, and
      // stop using the buffer
      set_status(p.status, MOE_DEV_TIMEOUT);
      ring_wait(bar, parity);
      break;
    }
    parity ^= 1u;
    for (int64_t w = 0; w < p.W; ++w) {
      // task w: groups 4w..4w+3, lane's 16 bytes of each half (see quant_kernel)
      const uint8_t* src = row + (4 * w * kGroup + lane * 8) * 2;
      const uint4 vA = (4 * w + half < p.G) ? *reinterpret_cast<const uint4*>(src)
                                            : make_uint4(0, 0, 0, 0);
      const uint4 vB = (4 * w + 2 + half < p.G) ? *reinterpret_cast<const uint4*>(src + 512)
                                                : make_uint4(0, 0, 0, 0);
      quant_task<SF_MODE, DISPATCH, SHARED>(p, t, w, vA, vB, lane);
    }
    // the buffer is read: refill it with this warp's next row
    __syncwarp();
    if (t + stride < p.T) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      if (lane == 0) bulk_row_load(row_s, p.hidden + (t + stride) * p.hs0, rowbytes, bar);
      __syncwarp();
    }
  }
}

}  // namespace moe

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
namespace moe_host {

using moe::StageParams;

size_t prepare_workspace_size(int64_t T, int64_t k, int64_t E) {
  const int64_t R = T * k;
  const int64_t B = (R + 1023) / 1024;
  size_t bytes = 256;                                   // completion counter
  bytes += (size_t)((B * E * 4 + 255) / 256) * 256;     // hist
  bytes += (size_t)((R * 4 + 255) / 256) * 256;         // local ranks
  return bytes;
}

template <typename Kernel>
static int64_t quant_grid(Kernel k, int64_t tasks) {
  // one wave of resident blocks: every warp loops over its share of tasks
  int64_t blocks = (tasks * 32 + 255) / 256;
  const int64_t cap = (int64_t)num_sms() * resident_blocks(reinterpret_cast<const void*>(k), 256);
  if (blocks > cap) blocks = cap;
  return blocks < 1 ? 1 : blocks;
}

// Long batches of rows up to 8192 values stream through shared memory
// (quant_ring_kernel); short ones spread each row over many warps
// (quant_kernel), which keeps a decode step's few rows from serialising.
constexpr int64_t kRingMinTokens = 1024;

static bool use_ring(const StageParams& p) { return p.K <= 8192 && p.T >= kRingMinTokens; }

// Row warps per block of a ring kernel: as many as the row buffers fit next
// to the load histogram in 227 KB (at most RING_MAX_WARPS), or up to four
// fewer when that deals the rows out in fuller rounds.  The rows go to
// blocks x warps in rounds, and a round takes about as long as the warps
// sharing an SM's bandwidth, so the cost is rounds x warps: 16,384 rows on
// 152 SMs take 8 rounds of 14 (112) or 9 of 12 (108).
static int ring_row_warps(int64_t T, int64_t K) {
  const size_t rowbytes = (size_t)(K * 2);
  const size_t hist = (size_t)moe::kLoadBins * sizeof(int);
  int wmax = (int)((227 * 1024 - 1024 - hist) / rowbytes);
  if (wmax > moe::RING_MAX_WARPS) wmax = moe::RING_MAX_WARPS;
  if (wmax < 1) wmax = 1;
  const int64_t sms = num_sms();
  int best = wmax;
  int64_t best_cost = (T + sms * wmax - 1) / (sms * wmax) * wmax;
  for (int w = wmax - 1; w >= 1 && w >= wmax - 4; --w) {
    const int64_t cost = (T + sms * w - 1) / (sms * w) * w;
    if (cost < best_cost) {
      best = w;
      best_cost = cost;
    }
  }
  return best;
}

template <typename Kernel>
static cudaError_t launch_ring(Kernel k, const StageParams& p, cudaStream_t s) {
  const size_t rowbytes = (size_t)(p.K * 2);
  const size_t hist = (size_t)moe::kLoadBins * sizeof(int);
  const int row_warps = ring_row_warps(p.T, p.K);
  const size_t smem = (size_t)row_warps * rowbytes + hist;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int64_t blocks = (p.T + row_warps - 1) / row_warps;
  if (blocks > num_sms()) blocks = num_sms();
  if (blocks < 1) blocks = 1;
  return launch_pdl(k, dim3((unsigned)blocks), dim3((row_warps + moe::RING_ROUTING_WARPS) * 32),
                    smem, s, p);
}

template <typename IdT, typename WT>
static moe_status_t launch_typed(StageParams& p, bool dispatch, int sf_mode, cudaStream_t s) {
  const int64_t tasks = p.T * p.W;
  const int threads = 256;
  const bool ring = use_ring(p);
  if (dispatch) {
    const int64_t R = p.T * p.top_k;
    if (!ring && R <= moe::kSmallRoutes && p.E * p.M_max < ((int64_t)1 << 31)) {
      // a decode-sized batch: routing and quantisation in one launch
      auto sk = sf_mode == MOE_SF_FP32
                    ? moe::small_dispatch_kernel<MOE_SF_FP32, IdT, WT, false>
                    : (p.shared_sf != nullptr
                           ? moe::small_dispatch_kernel<MOE_SF_UE8M0_PACKED, IdT, WT, true>
                           : moe::small_dispatch_kernel<MOE_SF_UE8M0_PACKED, IdT, WT, false>);
      const size_t ssm = (size_t)5 * p.E * sizeof(int32_t);
      cudaError_t le = launch_pdl(sk, dim3((unsigned)quant_grid(sk, tasks)), dim3(threads), ssm,
                                  s, p);
      if (le != cudaSuccess)
        return set_error(MOE_ERR_CUDA, "small_dispatch_kernel launch: %s", cudaGetErrorString(le));
      return MOE_OK;
    }
    const int64_t B = (R + 1023) / 1024;
    p.num_route_blocks = B;
    const size_t smem = (size_t)32 * p.E * sizeof(uint16_t);
    auto rk = moe::route_kernel<IdT, WT>;
    if (smem > 48 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(rk, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)smem);
      if (e != cudaSuccess)
        return set_error(MOE_ERR_CUDA, "route_kernel smem attribute: %s", cudaGetErrorString(e));
    }
    cudaError_t e = cudaMemsetAsync(p.done, 0, sizeof(uint32_t), s);
    if (e != cudaSuccess) return set_error(MOE_ERR_CUDA, "memset: %s", cudaGetErrorString(e));
    cudaError_t le = launch_pdl(rk, dim3((unsigned)B), dim3(1024), smem, s, p);
    if (le != cudaSuccess)
      return set_error(MOE_ERR_CUDA, "route_kernel launch: %s", cudaGetErrorString(le));
    // the shared-expert pages are a separate instantiation: even untaken,
    // their code costs the streaming loop ~10%
    if (ring) {
      auto qk = sf_mode == MOE_SF_FP32
                    ? moe::quant_ring_kernel<MOE_SF_FP32, false, true, IdT, WT, false>
                    : (p.shared_sf != nullptr
                           ? moe::quant_ring_kernel<MOE_SF_UE8M0_PACKED, false, true, IdT, WT, true>
                           : moe::quant_ring_kernel<MOE_SF_UE8M0_PACKED, false, true, IdT, WT,
                                                    false>);
      le = launch_ring(qk, p, s);
    } else {
      auto qk = sf_mode == MOE_SF_FP32
                    ? moe::quant_kernel<MOE_SF_FP32, false, true, IdT, WT, false>
                    : (p.shared_sf != nullptr
                           ? moe::quant_kernel<MOE_SF_UE8M0_PACKED, false, true, IdT, WT, true>
                           : moe::quant_kernel<MOE_SF_UE8M0_PACKED, false, true, IdT, WT, false>);
      le = launch_pdl(qk, dim3((unsigned)quant_grid(qk, tasks)), dim3(threads), 0, s, p);
    }
    if (le != cudaSuccess)
      return set_error(MOE_ERR_CUDA, "quant_kernel launch: %s", cudaGetErrorString(le));
  } else {
    switch (sf_mode) {
      case MOE_SF_NONE: {
        if (ring) {
          launch_ring(moe::quant_ring_kernel<MOE_SF_NONE, true, false, IdT, WT, false>, p, s);
        } else {
          auto qk = moe::quant_kernel<MOE_SF_NONE, true, false, IdT, WT, false>;
          launch_pdl(qk, dim3((unsigned)quant_grid(qk, tasks)), dim3(threads), 0, s, p);
        }
        break;
      }
      case MOE_SF_UE8M0_PACKED: {
        if (ring) {
          auto qk = p.shared_sf != nullptr
                        ? moe::quant_ring_kernel<MOE_SF_UE8M0_PACKED, true, false, IdT, WT, true>
                        : moe::quant_ring_kernel<MOE_SF_UE8M0_PACKED, true, false, IdT, WT, false>;
          launch_ring(qk, p, s);
        } else {
          auto qk = p.shared_sf != nullptr
                        ? moe::quant_kernel<MOE_SF_UE8M0_PACKED, true, false, IdT, WT, true>
                        : moe::quant_kernel<MOE_SF_UE8M0_PACKED, true, false, IdT, WT, false>;
          launch_pdl(qk, dim3((unsigned)quant_grid(qk, tasks)), dim3(threads), 0, s, p);
        }
        break;
      }
      default: {
        if (ring) {
          launch_ring(moe::quant_ring_kernel<MOE_SF_FP32, true, false, IdT, WT, false>, p, s);
        } else {
          auto qk = moe::quant_kernel<MOE_SF_FP32, true, false, IdT, WT, false>;
          launch_pdl(qk, dim3((unsigned)quant_grid(qk, tasks)), dim3(threads), 0, s, p);
        }
        break;
      }
    }
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(MOE_ERR_CUDA, "staging launch: %s", cudaGetErrorString(e));
  return MOE_OK;
}

moe_status_t launch_prepare(const moe_prepare_args_t* a, cudaStream_t s) {
  StageParams p{};
  p.T = a->num_tokens;
  p.K = a->hidden_size;
  p.top_k = a->top_k;
  p.G = a->hidden_size / 128;
  p.W = (p.G + 3) / 4;
  p.hidden = static_cast<const uint16_t*>(a->hidden);
  p.hs0 = a->hidden_stride0;
  p.ids = a->topk_ids;
  p.is0 = a->topk_ids_stride0;
  p.is1 = a->topk_ids_stride1;
  p.wts = a->topk_weights;
  p.ws0 = a->topk_weights_stride0;
  p.ws1 = a->topk_weights_stride1;
  p.pad = a->is_padding;
  p.ps0 = a->is_padding_stride0;
  p.x = static_cast<uint8_t*>(a->x);
  p.xs0 = a->x_stride0;
  p.x_sf = a->x_sf;
  p.sfs0 = a->x_sf_stride0;
  p.sfs1 = a->x_sf_stride1;
  p.shared_sf = a->shared_x_sf;
  p.ss0 = a->shared_x_sf_stride0;
  p.ss1 = a->shared_x_sf_stride1;
  p.sbm = a->shared_block_m > 0 ? a->shared_block_m : 1;
  p.sbm_aligned = (p.sbm + 127) / 128 * 128;
  p.sf_word = p.shared_sf != nullptr && p.ss1 == 1 && p.ss0 % 4 == 0 &&
              (reinterpret_cast<uintptr_t>(p.shared_sf) & 3u) == 0;
  p.ids_out = a->topk_idx_out;
  p.ios0 = a->topk_idx_out_stride0;
  p.ios1 = a->topk_idx_out_stride1;
  p.w_out = a->topk_weights_out;
  p.wos0 = a->topk_weights_out_stride0;
  p.wos1 = a->topk_weights_out_stride1;
  p.l2p = a->logical_to_physical;
  p.num_logical = a->num_logical;
  p.map_stride = a->map_stride;
  p.rep_count = a->logical_replica_count;
  p.load = a->expert_load;
  p.num_physical = a->num_physical;
  p.record = a->should_record;
  p.num_unpadded = a->num_unpadded_tokens;
  p.status = a->device_status;
  const bool dispatch = a->x_b != nullptr;
  if (dispatch) {
    p.E = a->num_experts;
    p.M_max = a->max_tokens_per_expert;
    p.x_b = static_cast<uint8_t*>(a->x_b);
    p.sf_b = static_cast<int32_t*>(a->sf_b);
    p.expert_num_tokens = a->expert_num_tokens;
    p.route_slot = a->route_slot;
    p.offsets = a->expert_offsets;
    const int64_t R = p.T * p.top_k;
    const int64_t B = (R + 1023) / 1024;
    char* ws = static_cast<char*>(a->workspace);
    p.done = reinterpret_cast<uint32_t*>(ws);
    p.hist = reinterpret_cast<int32_t*>(ws + 256);
    p.local_rank = reinterpret_cast<int32_t*>(ws + 256 + ((B * p.E * 4 + 255) / 256) * 256);
  }
  const bool ids64 = a->topk_ids_dtype == MOE_IDS_INT64;
  const bool wbf16 = a->topk_weights_dtype == MOE_WEIGHTS_BF16;
  if (ids64)
    return wbf16 ? launch_typed<int64_t, uint16_t>(p, dispatch, a->sf_mode, s)
                 : launch_typed<int64_t, float>(p, dispatch, a->sf_mode, s);
  return wbf16 ? launch_typed<int32_t, uint16_t>(p, dispatch, a->sf_mode, s)
               : launch_typed<int32_t, float>(p, dispatch, a->sf_mode, s);
}


template <typename IdT, typename WT>
static moe_status_t launch_nvfp4_typed(const moe::Nvfp4Params& q, const StageParams& p,
                                       cudaStream_t s) {
  // blocks per lane held in registers: the smallest of 4, 8, 14 (hidden 7168),
  // 16 that fits the row, else the row is streamed twice
  const int64_t nbl = (q.K / 16 + 31) / 32;
  auto pick = [&](auto fp8) {
    constexpr bool F = decltype(fp8)::value;
    return nbl <= 4    ? moe::nvfp4_kernel<IdT, WT, 4, F>
           : nbl <= 8  ? moe::nvfp4_kernel<IdT, WT, 8, F>
           : nbl <= 14 ? moe::nvfp4_kernel<IdT, WT, 14, F>
           : nbl <= 16 ? moe::nvfp4_kernel<IdT, WT, 16, F>
                       : moe::nvfp4_kernel<IdT, WT, 0, F>;
  };
  if (nbl <= 16) {
    // rows of up to 8192 values: streamed through shared memory, one block
    // of row warps and two routing warps per SM
    auto pick_ring = [&](auto fp8) {
      constexpr bool F = decltype(fp8)::value;
      return nbl <= 4    ? moe::nvfp4_ring_kernel<IdT, WT, 4, F>
             : nbl <= 8  ? moe::nvfp4_ring_kernel<IdT, WT, 8, F>
             : nbl <= 14 ? moe::nvfp4_ring_kernel<IdT, WT, 14, F>
                         : moe::nvfp4_ring_kernel<IdT, WT, 16, F>;
    };
    auto k = q.shared_q != nullptr ? pick_ring(std::true_type{}) : pick_ring(std::false_type{});
    // as many row buffers as fit next to the load histogram (and the static
    // 640 bytes) in 227 KB of shared memory
    const size_t rowbytes = (size_t)(q.K * 2);
    const size_t hist = (size_t)moe::kLoadBins * sizeof(int);
    const int row_warps = ring_row_warps(q.T, q.K);
    const size_t smem = (size_t)row_warps * rowbytes + hist;
    cudaError_t ae = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (ae != cudaSuccess)
      return set_error(MOE_ERR_CUDA, "nvfp4 smem attribute: %s", cudaGetErrorString(ae));
    int64_t blocks = (q.T + row_warps - 1) / row_warps;
    if (blocks > num_sms()) blocks = num_sms();
    if (blocks < 1) blocks = 1;
    cudaError_t e = launch_pdl(k, dim3((unsigned)blocks),
                               dim3((row_warps + moe::RING_ROUTING_WARPS) * 32), smem, s, q, p);
    if (e != cudaSuccess) return set_error(MOE_ERR_CUDA, "nvfp4 launch: %s", cudaGetErrorString(e));
    return MOE_OK;
  }
  auto k = q.shared_q != nullptr ? pick(std::true_type{}) : pick(std::false_type{});
  int64_t blocks = (q.T + 3) / 4;
  if (blocks < 1) blocks = 1;
  const int64_t cap = (int64_t)num_sms() * resident_blocks(reinterpret_cast<const void*>(k), 128);
  if (blocks > cap) blocks = cap;
  cudaError_t e = launch_pdl(k, dim3((unsigned)blocks), dim3(128), 0, s, q, p);
  if (e != cudaSuccess) return set_error(MOE_ERR_CUDA, "nvfp4 launch: %s", cudaGetErrorString(e));
  return MOE_OK;
}

moe_status_t launch_nvfp4(const moe_nvfp4_args_t* a, cudaStream_t s) {
  moe::Nvfp4Params q{};
  q.T = a->num_tokens;
  q.K = a->hidden_size;
  q.hidden = static_cast<const uint16_t*>(a->hidden);
  q.hs0 = a->hidden_stride0;
  q.x = a->x;
  q.xs0 = a->x_stride0;
  q.x_sf = reinterpret_cast<uint32_t*>(a->x_sf);
  q.sfs0 = a->x_sf_stride0;
  q.x_scales = a->x_scales;
  const bool fp8_shared = a->shared_x_dtype == MOE_SHARED_FP8;
  q.shared_x = fp8_shared ? nullptr : static_cast<uint16_t*>(a->shared_x);
  q.shared_q = fp8_shared ? static_cast<uint8_t*>(a->shared_x) : nullptr;
  q.shs0 = a->shared_x_stride0;
  q.shared_sf = a->shared_x_sf;
  q.ss0 = a->shared_x_sf_stride0;
  q.ss1 = a->shared_x_sf_stride1;
  q.sbm = a->shared_block_m > 0 ? a->shared_block_m : 1;
  q.sbm_aligned = (q.sbm + 127) / 128 * 128;
  q.w2gs = a->w2_global_scale;
  q.l2_alpha = a->l2_alpha;
  q.n_local = a->num_local_experts;
  q.l2s = a->l2_activation_scale;
  StageParams p{};
  p.T = a->num_tokens;
  p.K = a->hidden_size;
  p.top_k = a->top_k;
  p.ids = a->topk_ids;
  p.is0 = a->topk_ids_stride0;
  p.is1 = a->topk_ids_stride1;
  p.wts = a->topk_weights;
  p.ws0 = a->topk_weights_stride0;
  p.ws1 = a->topk_weights_stride1;
  p.pad = a->is_padding;
  p.ps0 = a->is_padding_stride0;
  p.ids_out = a->topk_idx_out;
  p.ios0 = a->topk_idx_out_stride0;
  p.ios1 = a->topk_idx_out_stride1;
  p.w_out = a->topk_weights_out;
  p.wos0 = a->topk_weights_out_stride0;
  p.wos1 = a->topk_weights_out_stride1;
  p.l2p = a->logical_to_physical;
  p.num_logical = a->num_logical;
  p.map_stride = a->map_stride;
  p.rep_count = a->logical_replica_count;
  p.load = a->expert_load;
  p.num_physical = a->num_physical;
  p.record = a->should_record;
  p.num_unpadded = a->num_unpadded_tokens;
  p.status = a->device_status;
  const bool i64 = a->topk_ids_dtype == MOE_IDS_INT64;
  const bool bf = a->topk_weights_dtype == MOE_WEIGHTS_BF16;
  if (i64) return bf ? launch_nvfp4_typed<int64_t, uint16_t>(q, p, s)
                     : launch_nvfp4_typed<int64_t, float>(q, p, s);
  return bf ? launch_nvfp4_typed<int32_t, uint16_t>(q, p, s)
            : launch_nvfp4_typed<int32_t, float>(q, p, s);
}

}  // namespace moe_host
