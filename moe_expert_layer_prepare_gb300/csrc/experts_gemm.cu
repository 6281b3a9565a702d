// Grouped-masked block-FP8 GEMMs of the batched MoE expert forward on sm_103a.
//
// Follows BatchedHummingGroupedExperts.apply and HummingExpertsBase
// (process_input / humming_forward / get_buffer_metas) on the page
// "vllm.model_executor.layers.fused_moe.experts.fused_humming_moe": the w13
// gate_up GEMM and the w2 down GEMM over the [E, M_max, K] layout, each
// expert's rows masked by expert_num_tokens, the activation (SiLU-and-mul)
// fused into the requantisation of the w2 input.
//
// One kernel template, two instances:
//   W13: h = x_b . w13^T (per expert), tile = 128 tokens x (128 gate + 128 up
//        columns of the same intermediate block); epilogue rounds h to bf16,
//        y = silu(gate) * up, 1x128 UE8M0 requant -> inter_q / inter_sf.
//   W2 : out = y_q . w2^T, tile = 128 tokens x 256 output columns, bf16
//        epilogue; optional split of the reduction with a deterministic
//        last-arriver reduce (partials summed in split order).
//
// Blackwell design
//   - persistent CTAs (one per SM), work units (expert, m-tile, n-tile,
//     split) enumerated on the device from expert_num_tokens, so empty
//     experts and tiles cost nothing and no host sync is needed;
//   - warp 0 issues TMA loads (128B-swizzled K-major tiles; the token tile
//     is loaded in 32-row boxes, only the rows that hold tokens);
//   - warp 1 owns TMEM (512 columns = two 128x256 fp32 accumulators) and
//     issues tcgen05.mma kind::f8f6f4 (E4M3 x E4M3 -> F32), one 128-wide K
//     slab per accumulator;
//   - warps 2..9 read each slab's partial product from TMEM (tcgen05.ld) and
//     fold it into fp32 registers with the slab's scale
//     2^(e_x - 127) * s_w[n/128, k/128]: the weight scales are arbitrary fp32
//     per 128x128 block, which the MMA's block-scale operand (UE8M0 only)
//     cannot carry, so the scale is applied per slab while the tensor core
//     works on the next slab in the other accumulator.
// Every wait is bounded (about 2 s); on expiry the CTA sets MOE_DEV_TIMEOUT,
// drains its copies and MMAs, frees TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdio>
#include <cstring>
#include <mutex>

#include "common.cuh"

namespace moe {

constexpr int BM = 128;          // tokens per tile (MMA M)
constexpr int BN = 256;          // MMA N
constexpr int BK = 128;          // K slab = one scale block
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK;              // 16 KB
constexpr int B_BYTES = BN * BK;              // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int A_BOX_ROWS = 32;
constexpr int NUM_THREADS = 384;              // 12 warps = 3 warpgroups
constexpr int EPI_WARP0 = 4;                  // warpgroups 1-2 are the epilogue
constexpr int EPI_WARPS = 8;
// Register split (setmaxnreg): the kernel is compiled for 168 registers per
// thread (384 x 168 = 64512); warpgroup 0 (TMA, MMA, the two scale-staging
// warps) drops and the two epilogue warpgroups rise.  The split is chosen per
// instantiation by what ptxas spills and what the GEMM then measures: the w2
// GEMM compiles spill-free at 56 / 224, the w13 GEMM spills least at 72 / 216
// (its fp32-scale form at 40 / 232).  Each sums to 128 x P + 256 x E <= 64512.
constexpr int LAUNCH_REGS = 168;
constexpr int producer_regs(bool w13, bool af32) { return !w13 ? 56 : (af32 ? 40 : 72); }
constexpr int epilogue_regs(bool w13, bool af32) { return !w13 ? 224 : (af32 ? 232 : 216); }
static_assert(128 * producer_regs(false, false) + 256 * epilogue_regs(false, false) <=
                  NUM_THREADS * LAUNCH_REGS, "register split exceeds the launch allocation");
static_assert(128 * producer_regs(true, false) + 256 * epilogue_regs(true, false) <=
                  NUM_THREADS * LAUNCH_REGS, "register split exceeds the launch allocation");
static_assert(128 * producer_regs(true, true) + 256 * epilogue_regs(true, true) <=
                  NUM_THREADS * LAUNCH_REGS, "register split exceeds the launch allocation");
constexpr int MAX_EXPERTS = 1024;
constexpr uint32_t TMEM_COLS = 512;
// Scale staging (UE8M0 activation scales): the two spare warps of warpgroup 0
// copy each unit's scales into shared memory, a window of up to SC_SLABS
// K slabs at a time, two windows in flight.
constexpr int SC_SLABS = 64;
constexpr int SC_WORDS = SC_SLABS / 4 + 1;   // exponent words of a window, any alignment
constexpr int SC_ROW = SC_WORDS;             // row stride in words (17: conflict-free reads)
constexpr int SC_THREADS = 64;               // warps 2 and 3

struct GemmParams {
  int E, M_max;
  int Kr;          // reduction length (K for w13, N for w2)
  int KB;          // Kr / 128
  int n_tiles;     // N/128 (w13) or ceil(K/256) (w2)
  int splits;      // reduction splits (w2 only)
  int N;           // intermediate size
  int K;           // hidden size
  int b_rows;      // rows of one expert in the B tensor (2N or K)
  const int32_t* expert_num_tokens;
  const int32_t* offsets;  // contiguous layout: [E+1] first row of each expert (nullable)
  const uint32_t* a_sf;  // packed UE8M0 words [E*M_max, Wa]; fp32 [E*M_max, Wa] when AF32
  int Wa;                // row stride of a_sf in 4-byte words
  const float* w_s;      // [E, b_rows/128, KB]
  // w13 outputs
  uint8_t* y_q;          // [E*M_max, N]
  uint8_t* y_sf_bytes;   // packed words viewed as bytes [E*M_max, 4*Wy]
  int Wy;
  uint16_t* h_dump;      // nullable bf16 [E*M_max, 2N]
  int yq_al32;           // y_q 32-byte aligned: 32-byte row stores
  // w2 outputs
  uint16_t* out;         // bf16 [E*M_max, K]
  int out_al32;          // out 32-byte aligned: 32-byte row stores
  float* partials;       // [splits, E*M_max, K]
  int32_t* counters;     // [(E * mt_max + E) * n_tiles]
  int mt_max;
  int32_t* zero_counters;  // w13 zeroes the next w2's counters
  int n_zero_counters;
  uint32_t* status;
};

// ------------------------------------------------------------------ PTX
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Limit of one pipeline wait in nanoseconds (2 s; the timeout test's build
// shortens it).
#ifndef MOE_WAIT_LIMIT_NS
#define MOE_WAIT_LIMIT_NS 2000000000ull
#endif

// Bounded wait: false when the CTA aborted or this wait exceeded the limit.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          uint32_t* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0u) {
      if (*abort_flag) return false;
      if (globaltimer() - t0 > (uint64_t)MOE_WAIT_LIMIT_NS) {
        *abort_flag = 1;
        set_status(status, MOE_DEV_TIMEOUT);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// One lane of the (converged) warp returns true.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred;
  asm volatile("{ .reg .pred p; elect.sync _|p, 0xffffffff; selp.u32 %0, 1, 0, p; }" : "=r"(pred));
  return pred != 0;
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (SBO), start address encoded >> 4, fixed 0b001 at bit 46.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;             // LBO (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;   // SBO
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;             // SWIZZLE_128B
  return d;
}

// Instruction descriptor: D f32, A/B e4m3, both K-major, N = 256, M = 128.
constexpr uint32_t kIdesc = (1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t)(BN >> 3) << 17) |
                            ((uint32_t)(BM >> 4) << 24);

__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0;"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p; }" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

#define TMEM_LD32(taddr, r)                                                                   \
  asm volatile(                                                                               \
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13," \
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"      \
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),   \
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),            \
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),         \
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),         \
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),         \
        "=r"(r[31])                                                                           \
      : "r"(taddr))

// 64 consecutive TMEM columns of this warp's 32 lanes into 64 registers.
#define TMEM_LD64(taddr, r)                                                              \
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x64.b32 {"                                \
               "%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,"                \
               "%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,"                \
               "%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"             \
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), \
                 "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), \
                 "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), \
                 "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), \
                 "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), \
                 "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), \
                 "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), \
                 "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), \
                 "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), \
                 "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), \
                 "=r"(r[61]), "=r"(r[62]), "=r"(r[63]) \
               : "r"(taddr))

// Wait for outstanding TMEM loads; the 64 destination registers are tied to
// the wait so that no use of them is scheduled before it.
#define TMEM_WAIT_PIN64(r)                                                               \
  asm volatile("tcgen05.wait::ld.sync.aligned;"                                         \
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), \
                 "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), \
                 "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), \
                 "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), \
                 "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), \
                 "+r"(r[31]), "+r"(r[32]), "+r"(r[33]), "+r"(r[34]), "+r"(r[35]), "+r"(r[36]), \
                 "+r"(r[37]), "+r"(r[38]), "+r"(r[39]), "+r"(r[40]), "+r"(r[41]), "+r"(r[42]), \
                 "+r"(r[43]), "+r"(r[44]), "+r"(r[45]), "+r"(r[46]), "+r"(r[47]), "+r"(r[48]), \
                 "+r"(r[49]), "+r"(r[50]), "+r"(r[51]), "+r"(r[52]), "+r"(r[53]), "+r"(r[54]), \
                 "+r"(r[55]), "+r"(r[56]), "+r"(r[57]), "+r"(r[58]), "+r"(r[59]), "+r"(r[60]), \
                 "+r"(r[61]), "+r"(r[62]), "+r"(r[63]) \
               :                                                                        \
               : "memory")

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Wait for outstanding TMEM loads; the 32 destination registers of the last
// load are read-write operands so that no use of them can move above the wait.
#define TMEM_WAIT_PIN32(r)                                                                      \
  asm volatile("tcgen05.wait::ld.sync.aligned;"                                                 \
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),        \
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),      \
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),  \
                 "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),  \
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),  \
                 "+r"(r[30]), "+r"(r[31])                                                       \
               :                                                                                \
               : "memory")

// dst[i] += r[i] * s for 32 columns with packed fp32x2 FMAs (round to nearest).
#define FMA32X2(dst, r, s)                                                            \
  _Pragma("unroll") for (int i_ = 0; i_ < 32; i_ += 2) {                              \
    const float2 d_ = __ffma2_rn(                                                     \
        make_float2(__uint_as_float((r)[i_]), __uint_as_float((r)[i_ + 1])),          \
        make_float2((s), (s)), make_float2((dst)[i_], (dst)[i_ + 1]));                \
    (dst)[i_] = d_.x;                                                                 \
    (dst)[i_ + 1] = d_.y;                                                             \
  }

// The epilogue's per-slab fold, in packed fp32x2 FMAs (measured against
// single FMAs on prefill: w13 -1.7%, w2 -4%).
#define FOLD32(dst, r, s) \
  { FMA32X2(dst, r, s); }

// ------------------------------------------------------------------ schedule
struct Unit {
  int e, mt, nt, ks, rows, kb0, kb1;
  int row0;  // first row of the tile in the [E*M_max, .] buffers
  int gmt;   // global m-tile index (split-K counters of the contiguous layout)
};

// Units are numbered expert by expert.  Inside an expert, w2 takes them
// m-tile-major (tile (mt, nt) at mt * n_tiles + nt) and w13 n-tile-major, so
// that the m-tiles sharing one w13 weight tile run side by side and the
// second and third reads of it hit L2 (measured: prefill w13 -2%, w2 +3% with
// the same order, so w2 keeps the other one).
template <bool W13>
__device__ __forceinline__ Unit decode_unit(const GemmParams& p, const int* prefix, int u,
                                            const int* cnt) {
  Unit w;
  const int per_mt = p.n_tiles * p.splits;
  const int mt_idx = u / per_mt;
  const int rem = u - mt_idx * per_mt;
  w.nt = rem / p.splits;
  w.ks = rem - w.nt * p.splits;
  int lo = 0, hi = p.E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= mt_idx) lo = mid; else hi = mid - 1;
  }
  w.e = lo;
  if constexpr (W13) {
    const int mt_e = prefix[lo + 1] - prefix[lo];
    const int l = u - prefix[lo] * per_mt;
    w.nt = l / (mt_e * p.splits);
    const int r2 = l - w.nt * (mt_e * p.splits);
    w.mt = r2 / p.splits;
    w.ks = r2 - w.mt * p.splits;
  } else {
    w.mt = mt_idx - prefix[lo];
  }
  w.rows = min(BM, cnt[lo] - w.mt * BM);
  w.row0 = (p.offsets != nullptr ? __ldg(p.offsets + lo) : lo * p.M_max) + w.mt * BM;
  w.gmt = prefix[lo] + w.mt;
  const int per = (p.KB + p.splits - 1) / p.splits;
  w.kb0 = w.ks * per;
  w.kb1 = min(p.KB, w.kb0 + per);
  return w;
}

// ------------------------------------------------------------------ kernel
template <bool W13, bool AF32 = false>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ GemmParams p,
                        const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  // bars: full[STAGES], empty[STAGES], tfull[2], tempty[2], mma_done, epi,
  //       sc_full[2], sc_empty[2]
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 10);
  int* s_abort = reinterpret_cast<int*>(tmem_holder + 1);
  int* s_flag = s_abort + 1;
  int* cnt = s_flag + 2;                 // [E]
  int* prefix = cnt + MAX_EXPERTS;       // [E+1]
  float* xamax = reinterpret_cast<float*>(prefix + MAX_EXPERTS + 4);  // [2][2][128]
  float* sc_w = xamax + 2 * 2 * BM;                                      // [2 windows][2][SC_SLABS]
  uint32_t* sc_a = reinterpret_cast<uint32_t*>(sc_w + 2 * 2 * SC_SLABS); // [2 windows][BM][SC_ROW]

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  volatile int* abort_flag = s_abort;

  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = smem_u32(bars + STAGES);
  const uint32_t tfull0 = smem_u32(bars + 2 * STAGES);
  const uint32_t tempty0 = smem_u32(bars + 2 * STAGES + 2);
  const uint32_t mma_done = smem_u32(bars + 2 * STAGES + 4);
  const uint32_t epi_bar = smem_u32(bars + 2 * STAGES + 5);
  const uint32_t sc_full0 = smem_u32(bars + 2 * STAGES + 6);
  const uint32_t sc_empty0 = smem_u32(bars + 2 * STAGES + 8);

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull0 + 8 * b, 1);
      mbar_init(tempty0 + 8 * b, EPI_WARPS);
    }
    mbar_init(mma_done, 1);
    mbar_init(epi_bar, EPI_WARPS);
    for (int b = 0; b < 2; ++b) {
      mbar_init(sc_full0 + 8 * b, SC_THREADS);
      mbar_init(sc_empty0 + 8 * b, EPI_WARPS);
    }
    *s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_holder)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // Everything above touches only this CTA's shared memory and TMEM; from
  // here on global memory written by the previous kernels is read.
  if (warp == 0 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
  }
  pdl_wait();
  pdl_launch_dependents();
  if (W13 && p.zero_counters != nullptr) {
    for (int i = blockIdx.x * NUM_THREADS + tid; i < p.n_zero_counters;
         i += gridDim.x * NUM_THREADS)
      p.zero_counters[i] = 0;
  }
  // Per-expert row counts and the exclusive prefix of m-tiles.
  for (int e = tid; e < p.E; e += NUM_THREADS) {
    int n;
    if (p.offsets == nullptr) {
      n = p.expert_num_tokens[e];
      n = n < 0 ? 0 : (n > p.M_max ? p.M_max : n);
    } else {
      // contiguous layout: rows [offsets[e], offsets[e+1]), kept inside the
      // E*M_max-row buffers whatever the offsets say
      const int64_t rows_total = (int64_t)p.E * p.M_max;
      const int64_t o0 = p.offsets[e], o1 = p.offsets[e + 1];
      n = (o0 < 0 || o1 <= o0 || o0 >= rows_total) ? 0 : (int)min(o1, rows_total) - (int)o0;
    }
    cnt[e] = n;
  }
  __syncthreads();
  if (warp == 0) {
    int running = 0;
    for (int base = 0; base < p.E; base += 32) {
      const int e = base + lane;
      int v = e < p.E ? (cnt[e] + BM - 1) / BM : 0;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xFFFFFFFFu, v, off);
        if (lane >= off) v += o;
      }
      if (e < p.E) prefix[e + 1] = running + v;
      running += __shfl_sync(0xFFFFFFFFu, v, 31);
    }
    if (lane == 0) prefix[0] = 0;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int total_units = prefix[p.E] * p.n_tiles * p.splits;

  if (warp < EPI_WARP0) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(producer_regs(W13, AF32)));
    // The producer and MMA loops run on all 32 lanes of their warp with
    // warp-uniform control flow, so every tcgen05 / TMA operand stays
    // warp-uniform; one elected lane issues each instruction.
    if (warp == 0) {
      // ---------------------------------------------------------------- TMA
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, issued_phase = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x) {
        const Unit w = decode_unit<W13>(p, prefix, u, cnt);
        const int a_row0 = w.row0;
        const int n_boxes = (w.rows + A_BOX_ROWS - 1) / A_BOX_ROWS;
        const uint32_t tx = (uint32_t)(n_boxes * A_BOX_ROWS * BK + B_BYTES);
        int b_row0, b_row1;
        if constexpr (W13) {
          b_row0 = w.e * p.b_rows + w.nt * 128;
          b_row1 = w.e * p.b_rows + p.N + w.nt * 128;
        } else {
          b_row0 = w.e * p.b_rows + w.nt * 256;
          b_row1 = b_row0 + 128;
        }
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          if (!__all_sync(0xFFFFFFFFu,
                          mbar_wait(empty0 + 8 * stage, phase ^ 1u, abort_flag, p.status))) {
            ok = false;
            break;
          }
          const uint32_t fb = full0 + 8 * stage;
          const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
          const uint32_t sb = sa + A_BYTES;
#ifdef MOE_TEST_WITHHOLD_STAGE
          // Failure-detection test builds only (the library build never sets
          // this): CTA 0 withholds the third stage of its first unit -- no
          // expect_tx and no copy, so no copy is ever left in flight -- and
          // the MMA warp's bounded wait on that stage runs out.
          const bool withhold = blockIdx.x == 0 && u == (int)blockIdx.x && kb == w.kb0 + 2;
#else
          constexpr bool withhold = false;
#endif
          if (!withhold) {
            if (elect_one()) {
              mbar_expect_tx(fb, tx);
              for (int i = 0; i < n_boxes; ++i)
                tma_load_2d(sa + i * A_BOX_ROWS * BK, &tmA, kb * BK, a_row0 + i * A_BOX_ROWS, fb);
              tma_load_2d(sb, &tmB, kb * BK, b_row0, fb);
              tma_load_2d(sb + 128 * BK, &tmB, kb * BK, b_row1, fb);
            }
            __syncwarp();
            issued_mask |= 1u << stage;
            issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Drain: every issued stage's copy must have landed before exit.
      for (int st = 0; st < STAGES; ++st) {
        if (issued_mask & (1u << st)) {
          volatile int never = 0;
          mbar_wait(full0 + 8 * st, (issued_phase >> st) & 1u, &never, p.status);
        }
      }
      __syncwarp();
    } else if (warp == 1) {
      // ---------------------------------------------------------------- MMA
      int stage = 0;
      uint32_t phase = 0;
      int ab = 0;
      uint32_t aphase = 0;
      bool ok = true;
      bool any = false;
      for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x) {
        const Unit w = decode_unit<W13>(p, prefix, u, cnt);
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          const bool ready = mbar_wait(tempty0 + 8 * ab, aphase ^ 1u, abort_flag, p.status) &&
                             mbar_wait(full0 + 8 * stage, phase, abort_flag, p.status);
          if (!__all_sync(0xFFFFFFFFu, ready)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
          const uint64_t adesc = sw128_desc(sa);
          const uint64_t bdesc = sw128_desc(sa + A_BYTES);
          const uint32_t d = tmem_base + (uint32_t)(ab * BN);
          if (elect_one()) {
#pragma unroll
            for (int k = 0; k < BK / 32; ++k)
              mma_f8(d, adesc + (uint64_t)(2 * k), bdesc + (uint64_t)(2 * k), k > 0 ? 1u : 0u);
            mma_commit(empty0 + 8 * stage);
            mma_commit(tfull0 + 8 * ab);
          }
          __syncwarp();
          any = true;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
          ab ^= 1;
          if (ab == 0) aphase ^= 1u;
        }
      }
      if (any) {
        // all MMAs of this CTA complete before TMEM is freed
        if (elect_one()) mma_commit(mma_done);
        __syncwarp();
        volatile int never = 0;
        mbar_wait(mma_done, 0, &never, p.status);
        __syncwarp();
      }
    } else if constexpr (!AF32) {
      // ---------------------------------------------------------- scale stager
      // Warps 2 and 3 walk the same units as the epilogue and copy, window by
      // window (up to SC_SLABS K slabs), the two weight-block scales of each
      // slab and the packed UE8M0 exponent words of the unit's rows into
      // shared memory, one window ahead of the epilogue.
      const int st = tid - 2 * 32;  // 0..63
      const int nblocks = p.b_rows / 128;
      int slot = 0;
      uint32_t sph = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x) {
        const Unit w = decode_unit<W13>(p, prefix, u, cnt);
        int nb0, nb1;
        if constexpr (W13) {
          nb0 = w.nt;
          nb1 = p.N / 128 + w.nt;
        } else {
          nb0 = 2 * w.nt;
          nb1 = 2 * w.nt + 1;
        }
        const float* ws0 = p.w_s + ((int64_t)w.e * nblocks + min(nb0, nblocks - 1)) * p.KB;
        const float* ws1 = p.w_s + ((int64_t)w.e * nblocks + min(nb1, nblocks - 1)) * p.KB;
        for (int wk0 = w.kb0; wk0 < w.kb1; wk0 += SC_SLABS) {
          const int nslab = min(w.kb1 - wk0, SC_SLABS);
          if (!__all_sync(0xFFFFFFFFu,
                          mbar_wait(sc_empty0 + 8 * slot, sph ^ 1u, abort_flag, p.status))) {
            ok = false;
            break;
          }
          float* dw = sc_w + slot * 2 * SC_SLABS;
          for (int j = st; j < nslab; j += SC_THREADS) {
            dw[j] = __ldg(ws0 + wk0 + j);
            dw[SC_SLABS + j] = __ldg(ws1 + wk0 + j);
          }
          const int word0 = wk0 >> 2;
          const int nwords = ((wk0 + nslab - 1) >> 2) - word0 + 1;
          uint32_t* da = sc_a + slot * BM * SC_ROW;
          for (int idx = st; idx < w.rows * nwords; idx += SC_THREADS) {
            const int r = idx / nwords;
            const int c = idx - r * nwords;
            da[r * SC_ROW + c] = __ldg(p.a_sf + (int64_t)(w.row0 + r) * p.Wa + word0 + c);
          }
          mbar_arrive(sc_full0 + 8 * slot);  // release: each thread's stores
          slot ^= 1;
          if (slot == 0) sph ^= 1u;
        }
      }
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(epilogue_regs(W13, AF32)));
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;                    // TMEM lane quarter
    const int h = (warp - EPI_WARP0) >> 2;     // column half
    const int row_local = q * 32 + lane;
    const uint32_t lane_addr = tmem_base + ((uint32_t)(q * 32) << 16);
    int ab = 0;
    uint32_t aphase = 0;
    int tp = 0;
    uint32_t epi_phase = 0;
    int sc_slot = 0;        // scale staging window in use, and its phase
    uint32_t sc_ph = 0;
    bool ok = true;
    const int64_t EM = (int64_t)p.E * p.M_max;
    // Bounded barrier of the eight epilogue warps (an mbarrier, so that an
    // aborted CTA can never hang in it).
    auto epi_sync = [&]() {
      __syncwarp();
      if (lane == 0) mbar_arrive(epi_bar);
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(epi_bar, epi_phase, abort_flag, p.status)))
        ok = false;
      epi_phase ^= 1u;
    };
    // TMEM column offsets of this thread's four 32-column groups.
    uint32_t cg[4];
#pragma unroll
    for (int c = 0; c < 4; ++c)
      cg[c] = W13 ? (uint32_t)((c < 2 ? 0 : 128) + h * 64 + (c & 1) * 32)
                  : (uint32_t)(h * 128 + c * 32);
    for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x) {
      const Unit w = decode_unit<W13>(p, prefix, u, cnt);
      const bool row_ok = row_local < w.rows;
      const bool warp_active = q * 32 < w.rows;   // warp-uniform
      const int64_t grow = (int64_t)w.row0 + row_local;
      float acc[128];
#pragma unroll
      for (int i = 0; i < 128; ++i) acc[i] = 0.0f;

      // One K slab: wait for its accumulator, read it from TMEM (two
      // 64-column loads, one wait each; W13: the gate half, then the up half)
      // and fold it into acc with the slab's scales; the accumulator is
      // released as soon as its second half is in registers.
#define FOLD_SLAB(S0, S1)                                                                     \
  {                                                                                           \
    if (!__all_sync(0xFFFFFFFFu, mbar_wait(tfull0 + 8 * ab, aphase, abort_flag, p.status))) { \
      ok = false;                                                                             \
      break;                                                                                  \
    }                                                                                         \
    if (warp_active) {                                                                        \
      tc_fence_after();                                                                       \
      const uint32_t base = lane_addr + (uint32_t)(ab * BN);                                  \
      uint32_t r64[64];                                                                       \
      TMEM_LD64(base + cg[0], r64);                                                           \
      TMEM_WAIT_PIN64(r64);                                                                   \
      FOLD32(acc + 0, r64, (S0));                                                             \
      FOLD32(acc + 32, r64 + 32, (S0));                                                       \
      TMEM_LD64(base + cg[2], r64);                                                           \
      TMEM_WAIT_PIN64(r64);                                                                   \
      tc_fence_before();                                                                      \
      __syncwarp();                                                                           \
      if (lane == 0) mbar_arrive(tempty0 + 8 * ab);                                           \
      FOLD32(acc + 64, r64, (S1));                                                            \
      FOLD32(acc + 96, r64 + 32, (S1));                                                       \
    } else {                                                                                  \
      __syncwarp();                                                                           \
      if (lane == 0) mbar_arrive(tempty0 + 8 * ab);                                           \
    }                                                                                         \
    ab ^= 1;                                                                                  \
    if (ab == 0) aphase ^= 1u;                                                                \
  }

      if constexpr (!AF32) {
        // UE8M0 activation scales: the scale stager has copied each window's
        // weight-block scales and this unit's exponent words to shared
        // memory; a slab's scale is two broadcast reads and this row's word.
        for (int wk0 = w.kb0; wk0 < w.kb1; wk0 += SC_SLABS) {
          const int wend = min(w.kb1, wk0 + SC_SLABS);
          if (!__all_sync(0xFFFFFFFFu,
                          mbar_wait(sc_full0 + 8 * sc_slot, sc_ph, abort_flag, p.status))) {
            ok = false;
            break;
          }
          const float* sw = sc_w + sc_slot * 2 * SC_SLABS + (W13 ? 0 : h * SC_SLABS);
          const uint32_t* srow = sc_a + (sc_slot * BM + row_local) * SC_ROW;
          const int word0 = wk0 >> 2;
          for (int kb = wk0; kb < wend; ++kb) {
            const uint32_t ea = (srow[(kb >> 2) - word0] >> (8 * (kb & 3))) & 0xFFu;
            const float sa = __uint_as_float(max(ea, 1u) << 23);
            const float s0 = sa * sw[kb - wk0];
            const float s1 = W13 ? sa * sw[SC_SLABS + kb - wk0] : s0;
            FOLD_SLAB(s0, s1)
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(sc_empty0 + 8 * sc_slot);
          sc_slot ^= 1;
          if (sc_slot == 0) sc_ph ^= 1u;
          if (!ok) break;
        }
      } else {
        // fp32 activation scales (a separate instantiation): the weight block
        // scales are the same for every row, so lane i holds slab i of a
        // 32-slab window (the next window fetched a window ahead) and each
        // slab takes its pair by shuffle; the row's fp32 scales run in a ring
        // four slabs ahead.
        int nb0, nb1;
        if constexpr (W13) {
          nb0 = w.nt;                         // gate block
          nb1 = p.N / 128 + w.nt;             // up block
        } else {
          nb0 = 2 * w.nt + h;
          nb1 = nb0;
        }
        const int nblocks = p.b_rows / 128;
        const float* ws0 = p.w_s + ((int64_t)w.e * nblocks + min(nb0, nblocks - 1)) * p.KB;
        const float* ws1 = p.w_s + ((int64_t)w.e * nblocks + min(nb1, nblocks - 1)) * p.KB;
        const float* afr = reinterpret_cast<const float*>(p.a_sf) + (row_ok ? grow : 0) * p.Wa;
        int wb = w.kb0;
        float wg_cur = wb + lane < w.kb1 ? __ldg(ws0 + wb + lane) : 0.0f;
        float wu_cur = wb + lane < w.kb1 ? __ldg(ws1 + wb + lane) : 0.0f;
        float wg_nxt = wb + 32 + lane < w.kb1 ? __ldg(ws0 + wb + 32 + lane) : 0.0f;
        float wu_nxt = wb + 32 + lane < w.kb1 ? __ldg(ws1 + wb + 32 + lane) : 0.0f;
        float af0 = 1.0f, af1 = 1.0f, af2 = 1.0f, af3 = 1.0f;
        if (row_ok) {
          af0 = __ldg(afr + w.kb0);
          if (w.kb0 + 1 < w.kb1) af1 = __ldg(afr + w.kb0 + 1);
          if (w.kb0 + 2 < w.kb1) af2 = __ldg(afr + w.kb0 + 2);
          if (w.kb0 + 3 < w.kb1) af3 = __ldg(afr + w.kb0 + 3);
        }
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          if (kb - wb == 32) {
            wb = kb;
            wg_cur = wg_nxt;
            wu_cur = wu_nxt;
            wg_nxt = wb + 32 + lane < w.kb1 ? __ldg(ws0 + wb + 32 + lane) : 0.0f;
            wu_nxt = wb + 32 + lane < w.kb1 ? __ldg(ws1 + wb + 32 + lane) : 0.0f;
          }
          const float sa = af0;
          af0 = af1;
          af1 = af2;
          af2 = af3;
          if (row_ok && kb + 4 < w.kb1) af3 = __ldg(afr + kb + 4);
          const float s0 = sa * __shfl_sync(0xFFFFFFFFu, wg_cur, kb - wb);
          const float s1 = sa * __shfl_sync(0xFFFFFFFFu, wu_cur, kb - wb);
          FOLD_SLAB(s0, s1)
        }
      }
#undef FOLD_SLAB
      if (!ok) break;

      if constexpr (W13) {
        // ---- h -> bf16, SiLU-and-mul, 1x128 UE8M0 requant
        const int n0 = w.nt * 128 + h * 64;
        if (p.h_dump != nullptr && row_ok) {
          uint16_t* hg = p.h_dump + grow * (int64_t)(2 * p.N) + n0;
          uint16_t* hu = hg + p.N;
#pragma unroll
          for (int i = 0; i < 64; i += 8) {
            uint4 vg, vu;
            vg.x = f32_to_bf16_bits(acc[i]) | (f32_to_bf16_bits(acc[i + 1]) << 16);
            vg.y = f32_to_bf16_bits(acc[i + 2]) | (f32_to_bf16_bits(acc[i + 3]) << 16);
            vg.z = f32_to_bf16_bits(acc[i + 4]) | (f32_to_bf16_bits(acc[i + 5]) << 16);
            vg.w = f32_to_bf16_bits(acc[i + 6]) | (f32_to_bf16_bits(acc[i + 7]) << 16);
            vu.x = f32_to_bf16_bits(acc[64 + i]) | (f32_to_bf16_bits(acc[64 + i + 1]) << 16);
            vu.y = f32_to_bf16_bits(acc[64 + i + 2]) | (f32_to_bf16_bits(acc[64 + i + 3]) << 16);
            vu.z = f32_to_bf16_bits(acc[64 + i + 4]) | (f32_to_bf16_bits(acc[64 + i + 5]) << 16);
            vu.w = f32_to_bf16_bits(acc[64 + i + 6]) | (f32_to_bf16_bits(acc[64 + i + 7]) << 16);
            st_v4(hg + i, vg);
            st_v4(hu + i, vu);
          }
        }
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          const float g = bf16_bits_to_f32(f32_to_bf16_bits(acc[i]));
          const float up = bf16_bits_to_f32(f32_to_bf16_bits(acc[64 + i]));
          const float silu = __fdividef(g, 1.0f + __expf(-fmaxf(g, -80.0f)));
          const float y = silu * up;
          acc[i] = y;
          amax = fmaxf(amax, fabsf(y));
        }
        xamax[(tp * 2 + h) * BM + row_local] = amax;
        epi_sync();
        amax = fmaxf(amax, xamax[(tp * 2 + (h ^ 1)) * BM + row_local]);
        tp ^= 1;
        const uint32_t code = ue8m0_exponent(amax);
        const float inv = ue8m0_inverse(code);
        if (row_ok) {
          uint8_t* dst = p.y_q + grow * (int64_t)p.N + n0;
          // the row's 64 codes: two 32-byte stores when y_q allows, else four
          // 16-byte ones (each thread writes its own row)
          if (p.yq_al32) {
#pragma unroll
            for (int i = 0; i < 64; i += 32) {
              uint32_t v[8];
#pragma unroll
              for (int j = 0; j < 8; ++j)
                v[j] = pack4_e4m3(acc[i + 4 * j] * inv, acc[i + 4 * j + 1] * inv,
                                  acc[i + 4 * j + 2] * inv, acc[i + 4 * j + 3] * inv);
              st_v8(dst + i, v);
            }
          } else {
#pragma unroll
            for (int i = 0; i < 64; i += 16) {
              uint4 v;
              v.x = pack4_e4m3(acc[i] * inv, acc[i + 1] * inv, acc[i + 2] * inv, acc[i + 3] * inv);
              v.y = pack4_e4m3(acc[i + 4] * inv, acc[i + 5] * inv, acc[i + 6] * inv,
                               acc[i + 7] * inv);
              v.z = pack4_e4m3(acc[i + 8] * inv, acc[i + 9] * inv, acc[i + 10] * inv,
                               acc[i + 11] * inv);
              v.w = pack4_e4m3(acc[i + 12] * inv, acc[i + 13] * inv, acc[i + 14] * inv,
                               acc[i + 15] * inv);
              st_v4(dst + i, v);
            }
          }
          if (h == 0) p.y_sf_bytes[grow * (int64_t)(4 * p.Wy) + w.nt] = (uint8_t)code;
        }
      } else {
        // ---- bf16 output (optionally through split partials)
        const int c0 = w.nt * 256 + h * 128;
        const bool cols_ok = c0 < p.K;
        if (p.splits == 1) {
          if (row_ok && cols_ok) {
            uint16_t* dst = p.out + grow * (int64_t)p.K + c0;
            // Each thread writes its own row, so a warp's store touches 32
            // rows; 32-byte stores fill whole sectors and halve the store
            // instructions (prefill w2 -10% against 16-byte stores).
            if (p.out_al32) {
#pragma unroll
              for (int i = 0; i < 128; i += 16) {
                uint32_t v[8];
#pragma unroll
                for (int j = 0; j < 8; ++j)
                  v[j] = f32_to_bf16_bits(acc[i + 2 * j]) |
                         (f32_to_bf16_bits(acc[i + 2 * j + 1]) << 16);
                st_v8(dst + i, v);
              }
            } else {
#pragma unroll
              for (int i = 0; i < 128; i += 8) {
                uint4 v;
                v.x = f32_to_bf16_bits(acc[i]) | (f32_to_bf16_bits(acc[i + 1]) << 16);
                v.y = f32_to_bf16_bits(acc[i + 2]) | (f32_to_bf16_bits(acc[i + 3]) << 16);
                v.z = f32_to_bf16_bits(acc[i + 4]) | (f32_to_bf16_bits(acc[i + 5]) << 16);
                v.w = f32_to_bf16_bits(acc[i + 6]) | (f32_to_bf16_bits(acc[i + 7]) << 16);
                st_v4(dst + i, v);
              }
            }
          }
        } else {
          if (row_ok && cols_ok) {
            float* dst = p.partials + ((int64_t)w.ks * EM + grow) * p.K + c0;
#pragma unroll
            for (int i = 0; i < 128; i += 4)
              st_v4(dst + i, make_uint4(__float_as_uint(acc[i]), __float_as_uint(acc[i + 1]),
                                        __float_as_uint(acc[i + 2]), __float_as_uint(acc[i + 3])));
          }
          __threadfence();
          epi_sync();
          const int64_t ctr_row =
              p.offsets != nullptr ? (int64_t)w.gmt : (int64_t)w.e * p.mt_max + w.mt;
          int32_t* ctr = p.counters + ctr_row * p.n_tiles + w.nt;
          if (tid == EPI_WARP0 * 32) {
            const int prev = atomicAdd(ctr, 1);
            *s_flag = (prev == p.splits - 1) ? 1 : 0;
          }
          epi_sync();
          if (*s_flag) {
            __threadfence();
            if (row_ok && cols_ok) {
              // partials are summed in split order, 32 columns at a time
              uint16_t* dst = p.out + grow * (int64_t)p.K + c0;
#pragma unroll 1
              for (int c = 0; c < 128; c += 32) {
                float sum[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) sum[i] = 0.0f;
                for (int s = 0; s < p.splits; ++s) {
                  const float* src = p.partials + ((int64_t)s * EM + grow) * p.K + c0 + c;
#pragma unroll
                  for (int i = 0; i < 32; i += 4) {
                    const float4 v = __ldcg(reinterpret_cast<const float4*>(src + i));
                    sum[i] += v.x;
                    sum[i + 1] += v.y;
                    sum[i + 2] += v.z;
                    sum[i + 3] += v.w;
                  }
                }
#pragma unroll
                for (int i = 0; i < 32; i += 8) {
                  uint4 v;
                  v.x = f32_to_bf16_bits(sum[i]) | (f32_to_bf16_bits(sum[i + 1]) << 16);
                  v.y = f32_to_bf16_bits(sum[i + 2]) | (f32_to_bf16_bits(sum[i + 3]) << 16);
                  v.z = f32_to_bf16_bits(sum[i + 4]) | (f32_to_bf16_bits(sum[i + 5]) << 16);
                  v.w = f32_to_bf16_bits(sum[i + 6]) | (f32_to_bf16_bits(sum[i + 7]) << 16);
                  st_v4(dst + c + i, v);
                }
              }
            }
            if (tid == EPI_WARP0 * 32) *ctr = 0;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(TMEM_COLS)
                 : "memory");
  }
}

}  // namespace moe

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
namespace moe_host {

using moe::GemmParams;

static PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// 2-D fp8 tensor [rows, cols] (row pitch = cols bytes), box [box_rows, 128].
static bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                     uint32_t box_rows) {
  auto enc = get_encode();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides,
                   box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

static int64_t est_mtiles(int64_t E, int64_t M_max, int64_t vsm) {
  const int64_t mt_per = (M_max + 127) / 128;
  const int64_t cap = E * mt_per;
  if (vsm <= 0) return cap;
  int64_t est = (vsm < E ? vsm : E) + (M_max > 128 ? vsm / 128 : 0);
  return est < cap ? est : cap;
}

// Reduction splits of the w2 GEMM.  A split costs every unit its partial-sum
// stores, a fence and a tile counter, which stalls the CTA's MMA pipeline at
// each unit end; measured, 3 splits of 64 decode tiles (K = 2048) ran 19%
// slower than no split and 7 splits of Mixtral's 128 tiles 2.4x slower.  So
// the reduction is split only when the tiles leave most SMs idle (fewer than
// a quarter of them), with enough splits to cover ~90% of the SMs, at least 4
// slabs each, every split non-empty.
static int choose_splits(int64_t units_base, int KB, int sms) {
  if (units_base <= 0 || units_base * 4 >= (int64_t)sms) return 1;
  int64_t want = ((int64_t)sms * 9 / 10 + units_base - 1) / units_base;
  int sp = (int)(want > 16 ? 16 : want);
  while (sp > 1) {
    const int per = (KB + sp - 1) / sp;
    if (per >= 4 && (int64_t)(sp - 1) * per < KB) break;
    --sp;
  }
  return sp < 1 ? 1 : sp;
}

static int w2_splits(int64_t E, int64_t M_max, int64_t K, int64_t N, int64_t vsm) {
  const int64_t nt = (K + 255) / 256;
  return choose_splits(est_mtiles(E, M_max, vsm) * nt, (int)(N / 128), num_sms());
}

size_t experts_workspace_size(int64_t E, int64_t M_max, int64_t K, int64_t N, int64_t vsm,
                              int which) {
  const int64_t EM = E * M_max;
  if (which == 13) {
    const int64_t Wy = (N / 128 + 3) / 4;
    return (size_t)(((EM * N + 255) / 256) * 256 + ((EM * Wy * 4 + 255) / 256) * 256);
  }
  const int S = w2_splits(E, M_max, K, N, vsm);
  const int64_t nt = (K + 255) / 256;
  const int64_t mt_max = (M_max + 127) / 128;
  size_t bytes = (size_t)((((E * mt_max + E) * nt * 4) + 255) / 256) * 256;
  if (S > 1) bytes += (size_t)S * EM * K * 4;
  return bytes;
}

static size_t gemm_smem_bytes() {
  return 1024 + (size_t)moe::STAGES * moe::STAGE_BYTES + 256 +
         4 * (4 + 2 * moe::MAX_EXPERTS + 8) + 4 * 2 * 2 * moe::BM +
         4 * 2 * 2 * moe::SC_SLABS + 4 * 2 * moe::BM * moe::SC_ROW;
}

// Per-device set-up of the GEMM kernels: the dynamic shared-memory limit is
// a per-device function attribute, and the in-kernel register split assumes
// the launch allocation checked here.  Done once per device, under a lock, so
// that concurrent first calls and calls on several devices are all covered.
static moe_status_t prepare_kernels(size_t smem) {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static bool done[kMaxDevices] = {};
  int dev = -1;
  cudaError_t ge = cudaGetDevice(&dev);
  if (ge != cudaSuccess) return set_error(MOE_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(ge));
  if (dev < 0 || dev >= kMaxDevices)
    return set_error(MOE_ERR_UNSUPPORTED, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lock(mu);
  if (done[dev]) return MOE_OK;
  const void* kernels[3] = {reinterpret_cast<const void*>(moe::grouped_gemm_kernel<true>),
                            reinterpret_cast<const void*>(moe::grouped_gemm_kernel<false>),
                            reinterpret_cast<const void*>(moe::grouped_gemm_kernel<true, true>)};
  for (const void* k : kernels) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
      return set_error(MOE_ERR_CUDA, "GEMM smem attribute: %s", cudaGetErrorString(e));
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, k) != cudaSuccess)
      return set_error(MOE_ERR_CUDA, "cudaFuncGetAttributes failed for a GEMM kernel");
    if (fa.numRegs != moe::LAUNCH_REGS)
      return set_error(MOE_ERR_UNSUPPORTED,
                       "a GEMM kernel was built with %d registers per thread; the register "
                       "split needs exactly %d", fa.numRegs, moe::LAUNCH_REGS);
  }
  done[dev] = true;
  return MOE_OK;
}

moe_status_t launch_experts(const moe_experts_args_t* a, cudaStream_t s) {
  const int64_t E = a->num_experts, M = a->max_tokens_per_expert;
  const int64_t K = a->hidden_size, N = a->intermediate_size;
  const int64_t EM = E * M;
  if (E > moe::MAX_EXPERTS)
    return set_error(MOE_ERR_UNSUPPORTED, "at most %d experts", moe::MAX_EXPERTS);
  if (EM * (2 * N > K ? 2 * N : K) > ((int64_t)1 << 31) * 127 || E * 2 * N >= ((int64_t)1 << 31) ||
      E * K >= ((int64_t)1 << 31) || EM >= ((int64_t)1 << 31))
    return set_error(MOE_ERR_UNSUPPORTED, "problem too large for 32-bit tile coordinates");
  const int stages = a->stages == 0 ? MOE_STAGE_ALL : a->stages;
  const int64_t Wy = (N / 128 + 3) / 4;
  uint8_t* inter_q = static_cast<uint8_t*>(a->inter_q);
  uint32_t* inter_sf = static_cast<uint32_t*>(a->inter_sf);
  if (inter_q == nullptr) {
    char* ws = static_cast<char*>(a->workspace13);
    inter_q = reinterpret_cast<uint8_t*>(ws);
    inter_sf = reinterpret_cast<uint32_t*>(ws + ((EM * N + 255) / 256) * 256);
  }
  const int S = w2_splits(E, M, K, N, a->valid_shape_m);
  const int64_t nt2 = (K + 255) / 256;
  const int64_t mt_max = (M + 127) / 128;
  int32_t* counters = nullptr;
  float* partials = nullptr;
  if (stages & MOE_STAGE_W2) {
    char* ws2 = static_cast<char*>(a->workspace2);
    counters = reinterpret_cast<int32_t*>(ws2);
    partials = reinterpret_cast<float*>(ws2 + (((E * mt_max + E) * nt2 * 4 + 255) / 256) * 256);
  }
  const size_t smem = gemm_smem_bytes();
  const int sms = num_sms();
  {
    moe_status_t st = prepare_kernels(smem);
    if (st != MOE_OK) return st;
  }
  // Upper bound of the work units: every expert full.  Persistent grid.
  // (the contiguous layout has at most E + E*M/128 m-tiles)
  const int64_t mt_cap = E * mt_max + E;

  if (stages & MOE_STAGE_W13) {
    GemmParams p{};
    p.E = (int)E;
    p.M_max = (int)M;
    p.Kr = (int)K;
    p.KB = (int)(K / 128);
    p.n_tiles = (int)(N / 128);
    p.splits = 1;
    p.N = (int)N;
    p.K = (int)K;
    p.b_rows = (int)(2 * N);
    p.expert_num_tokens = a->expert_num_tokens;
    p.offsets = a->expert_offsets;
    p.a_sf = static_cast<const uint32_t*>(a->a_scale);
    const bool af32 = a->a_scale_mode == MOE_SF_FP32;
    p.Wa = af32 ? (int)(K / 128) : (int)((K / 128 + 3) / 4);
    p.w_s = a->w13_scale;
    p.y_q = inter_q;
    // rows of N bytes (N a multiple of 128) and column blocks of 64 bytes
    p.yq_al32 = (reinterpret_cast<uintptr_t>(inter_q) & 31u) == 0 ? 1 : 0;
    p.y_sf_bytes = reinterpret_cast<uint8_t*>(inter_sf);
    p.Wy = (int)Wy;
    p.h_dump = static_cast<uint16_t*>(a->gate_up_dump);
    p.mt_max = (int)mt_max;
    p.status = a->device_status;
    if ((stages & MOE_STAGE_W2) && S > 1) {
      p.zero_counters = counters;
      p.n_zero_counters = (int)((E * mt_max + E) * nt2);
    }
    CUtensorMap tA, tB;
    if (!make_map(&tA, a->hidden, (uint64_t)EM, (uint64_t)K, moe::A_BOX_ROWS) ||
        !make_map(&tB, a->w13, (uint64_t)(E * 2 * N), (uint64_t)K, 128))
      return set_error(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed for the w13 operands");
    const int64_t units = mt_cap * p.n_tiles;
    const int grid = (int)(units < sms ? (units < 1 ? 1 : units) : sms);
    cudaError_t e =
        af32 ? launch_pdl(moe::grouped_gemm_kernel<true, true>, dim3(grid),
                          dim3(moe::NUM_THREADS), smem, s, p, tA, tB)
             : launch_pdl(moe::grouped_gemm_kernel<true>, dim3(grid), dim3(moe::NUM_THREADS),
                          smem, s, p, tA, tB);
    if (e != cudaSuccess) return set_error(MOE_ERR_CUDA, "w13 launch: %s", cudaGetErrorString(e));
  }
  if (stages & MOE_STAGE_W2) {
    GemmParams p{};
    p.E = (int)E;
    p.M_max = (int)M;
    p.Kr = (int)N;
    p.KB = (int)(N / 128);
    p.n_tiles = (int)nt2;
    p.splits = S;
    p.N = (int)N;
    p.K = (int)K;
    p.b_rows = (int)K;
    p.expert_num_tokens = a->expert_num_tokens;
    p.offsets = a->expert_offsets;
    p.a_sf = inter_sf;
    p.Wa = (int)Wy;
    p.w_s = a->w2_scale;
    p.out = static_cast<uint16_t*>(a->output);
    // rows of 2K bytes (K a multiple of 128) and column blocks of 256 bytes
    p.out_al32 = (reinterpret_cast<uintptr_t>(a->output) & 31u) == 0 ? 1 : 0;
    p.partials = partials;
    p.counters = counters;
    p.mt_max = (int)mt_max;
    p.status = a->device_status;
    CUtensorMap tA, tB;
    if (!make_map(&tA, inter_q, (uint64_t)EM, (uint64_t)N, moe::A_BOX_ROWS) ||
        !make_map(&tB, a->w2, (uint64_t)(E * K), (uint64_t)N, 128))
      return set_error(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed for the w2 operands");
    const int64_t units = mt_cap * nt2 * S;
    const int grid = (int)(units < sms ? (units < 1 ? 1 : units) : sms);
    cudaError_t e = launch_pdl(moe::grouped_gemm_kernel<false>, dim3(grid), dim3(moe::NUM_THREADS),
                               smem, s, p, tA, tB);
    if (e != cudaSuccess) return set_error(MOE_ERR_CUDA, "w2 launch: %s", cudaGetErrorString(e));
  }
  return MOE_OK;
}

}  // namespace moe_host
