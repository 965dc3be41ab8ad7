// moe_internal.cuh -- device helpers and launcher declarations shared by the
// CUDA translation units of libmoe.so. Internal: not part of the C ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// ---------------------------------------------------------------------------
// Launch parameter blocks (host fills, kernels read by value).
// ---------------------------------------------------------------------------

struct LayoutParams {
  const int32_t* topk_idx;
  int32_t* tokens_per_expert;
  int32_t* tokens_per_rank;
  uint8_t* is_token_in_rank;
  int32_t* expert_offset;
  int32_t* rank_offset;
  int32_t* slot_of;
  int32_t* src_of_slot;  // may be null
  int32_t* status;       // workspace status word
  int32_t* chunk_hist;   // [chunks][E] per-chunk expert counts
  int32_t* chunk_rank;   // [chunks][R] per-chunk token-in-rank counts
  int32_t* chunk_flag;   // [chunks] invalid-id flags
  int num_tokens, topk, num_experts, num_ranks, experts_per_rank;
  int tokens_per_chunk, num_chunks;
  // The per-rank receive layout (moe_layout_ranks), computed by the cluster
  // kernel when send_head is set; null otherwise.
  int32_t* send_head = nullptr;               // [N, R]
  int32_t* recv_src_idx = nullptr;            // [N * R], may be null
  int32_t* recv_offset = nullptr;             // [R + 1]
  int32_t* recv_tokens_per_expert = nullptr;  // [E]
  int expert_alignment = 1;
  // The fixed-capacity, expert-major layout (moe_layout_ll), computed by the
  // cluster kernel when ll_slot_of is set; null otherwise.
  int32_t* ll_slot_of = nullptr;    // [N, k]
  int32_t* src_info = nullptr;      // [E, ll_capacity]
  int64_t* layout_range = nullptr;  // [E, R]
  int32_t* recv_count = nullptr;    // [E]
  int64_t ll_capacity = 0;          // R * max_tokens_per_rank
  int ll_tokens_per_rank = 0;       // T = N / R
};

struct DispatchParams {
  const int32_t* topk_idx;
  const float* topk_weights;
  const uint8_t* hidden;  // bf16 rows or raw payload rows
  const uint8_t* scales;  // raw scale rows (RAW only)
  const int32_t* slot_of;
  uint8_t* records;
  int64_t record_capacity;  // records the caller's buffer holds
  int num_tokens, topk, hidden_size;
  int in_row_bytes;   // bytes of one hidden row
  int in_scale_bytes; // bytes of one raw scale row (RAW)
  // record layout
  int record_bytes, off_ids, off_weights, off_payload, off_scales, payload_bytes, scale_bytes;
};

struct CombineParams {
  const uint8_t* expert_out;
  int64_t expert_out_rows;
  const int32_t* topk_idx;
  const float* topk_weights;
  const int32_t* slot_of;
  uint8_t* out;
  int num_tokens, topk, hidden_size, num_ranks, experts_per_rank;
  int group_by_rank;  // 1: TOPK_RANKS, 0: TOPK
};

struct CombineNormParams {
  CombineParams c;  // expert rows (or rank partials), pairs, shapes; c.out unused
  int mode;         // MOE_COMBINE_TOPK, MOE_COMBINE_RANKS or MOE_COMBINE_TOPK_RANKS
  const uint8_t* residual_in;  // bf16 [N, H]
  const uint8_t* gamma;        // bf16 [H]
  uint8_t* normed_out;         // bf16 [N, H]
  uint8_t* residual_out;       // bf16 [N, H]
  float eps;
};

struct RankLayoutParams {
  const uint8_t* is_token_in_rank;  // [N, R]
  const int32_t* tokens_per_rank;   // [R]
  const int32_t* tokens_per_expert; // [E]
  int32_t* send_head;               // [N, R]
  int32_t* recv_src_idx;            // [N * R], may be null
  int32_t* recv_offset;             // [R + 1]
  int32_t* recv_tokens_per_expert;  // [E]
  int num_tokens, num_ranks, num_experts, expert_alignment;
};

struct RankCombineParams {
  const uint8_t* recv_out;  // bf16 [rows, H]
  int64_t rows;
  const int32_t* send_head; // [N, R]
  uint8_t* out;             // bf16 [N, H]
  int num_tokens, num_ranks, hidden_size;
};

struct LlLayoutParams {
  const int32_t* topk_idx;       // [N, k]
  const int32_t* slot_of;        // [N, k]
  const int32_t* expert_offset;  // [E + 1]
  const int32_t* src_of_slot;    // [N * k]
  int32_t* ll_slot_of;           // [N, k]  e * capacity + position, or -1
  int32_t* src_info;             // [E, capacity]
  int64_t* layout_range;         // [E, R]  begin << 32 | count
  int32_t* recv_count;           // [E]
  int64_t capacity;              // R * max_tokens_per_rank
  int num_tokens, topk, num_experts, num_ranks;
};

struct CombineBwdParams {
  const uint8_t* grad_out;     // bf16 [N, H]
  const float* topk_weights;   // [N, k]
  const int32_t* slot_of;      // [N, k]
  const uint8_t* expert_out;   // bf16 [rows, H], null: no weight gradient
  int64_t rows;
  uint8_t* grad_expert_out;    // bf16 [rows, H]
  float* grad_weights;         // [N, k], used with expert_out
  int num_tokens, topk, hidden_size;
};

struct RankCombineBwdParams {
  const uint8_t* grad_out;  // bf16 [N, H]
  const int32_t* send_head; // [N, R]
  uint8_t* grad_recv;       // bf16 [rows, H]
  int64_t rows;
  int num_tokens, num_ranks, hidden_size;
};

// Programmatic dependent launch. Every kernel of this library begins with
// pdl_wait() -- griddepcontrol.wait: until the previous kernel in the stream
// has completed and its memory operations are visible -- before its first
// access to global memory, and then calls pdl_trigger() so that the next
// kernel's blocks may be scheduled while this one drains. Launched through
// launch_pdl (programmatic stream serialization), a kernel can thus be
// resident before its predecessor ends, which hides the launch gap; launched
// without it, both instructions do nothing. Setting the environment variable
// MOE_PDL=0 launches every kernel in plain stream order.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

bool pdl_enabled();

// The current device's index and SM count, looked up once per device
// (thread-safe); false if the device cannot be queried.
bool current_device(int* dev, int* sms);

// Raises fn's dynamic shared memory limit to at least `bytes` on the current
// device; the attribute is set only when a launch needs more than before
// (thread-safe).
cudaError_t ensure_dynamic_smem(const void* fn, size_t bytes);

// cudaLaunchKernelExC with the programmatic-serialization attribute (when
// enabled) and an optional cluster size (cluster_x > 0).
cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       void** args, unsigned cluster_x = 0);

// Workspace carving shared by moe_workspace_size and moe_layout.
constexpr int kLayoutTokensPerChunk = 128;
size_t layout_workspace_bytes(int num_tokens, int num_experts, int num_ranks);

// Launchers (return cudaError_t of the launch).
// extra_done (may be null) is set when the launch also computed the receive
// layout of p.send_head or the fixed-capacity layout of p.ll_slot_of;
// otherwise the caller runs launch_rank_layout or launch_ll_layout.
cudaError_t launch_layout(const LayoutParams& p, cudaStream_t s, bool* extra_done = nullptr);
// after_layout: the previous kernel on s is this library's layout kernel,
// launched by the same call (moe_layout_dispatch), so the row work may start
// before it ends.
cudaError_t launch_dispatch(const DispatchParams& p, int in_kind, int out_kind, cudaStream_t s,
                            bool after_layout = false);
cudaError_t launch_combine_topk(const CombineParams& p, cudaStream_t s);
cudaError_t launch_combine_ranks(const uint8_t* partials, uint8_t* out, int64_t rows,
                                 int hidden_size, int num_ranks, cudaStream_t s);
cudaError_t launch_combine_norm(const CombineNormParams& p, cudaStream_t s);
// The device status word of the kernels with bounded waits (MOE_OK, or
// MOE_ERR_TIMEOUT once a wait gave up); synchronous. clear: reset it to MOE_OK.
int read_device_status(int32_t* out, bool clear);
// The budget of the bounded waits for launches from now on (ns; 0 = the
// default kWaitLimitNs; clamped to it).
void set_wait_limit_ns(uint64_t ns);
cudaError_t launch_slots(bool pack, const void* const* src, void* const* dst,
                         const moe_slot_desc_t* d, const int64_t* offsets, int64_t slot_bytes,
                         cudaStream_t s);
cudaError_t launch_rank_layout(const RankLayoutParams& p, cudaStream_t s);
// moe_layout_dispatch of a small routing (at most 2048 pairs) as one kernel
// that computes the layout in every block; fits() says whether it applies
// (MOE_FUSED_LAYOUT=n in the environment lowers the pair limit; 0 turns the
// kernel off).
bool layout_dispatch_small_fits(const DispatchParams& p, int out_kind, int num_experts);
cudaError_t launch_layout_dispatch_small(const DispatchParams& p, const LayoutParams& lp, int out_kind,
                                         cudaStream_t s);
cudaError_t launch_dispatch_ranks(const DispatchParams& p, int out_kind, const int32_t* send_head,
                                  int num_ranks, int experts_per_rank, cudaStream_t s);
cudaError_t launch_combine_gather_ranks(const RankCombineParams& p, cudaStream_t s);
cudaError_t launch_ll_layout(const LlLayoutParams& p, cudaStream_t s);
cudaError_t launch_combine_backward(const CombineBwdParams& p, cudaStream_t s);
cudaError_t launch_gather_ranks_backward(const RankCombineBwdParams& p, cudaStream_t s);
// after_layout (as in launch_dispatch): the previous kernel on s is the same
// call's layout, so the payload may be built before it ends.
cudaError_t launch_dispatch_packed(const DispatchParams& p, int out_kind, uint8_t* x_out,
                                   uint8_t* scales_out, int64_t rows, cudaStream_t s, bool after_layout = false);
cudaError_t launch_mask_topk_ids(int32_t* ids, int64_t total, int topk, const int32_t* num_actual,
                                 cudaStream_t s);
constexpr int kMaxHiddenNorm = 16384;

#ifdef __CUDACC__

// ---------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------

__device__ __forceinline__ unsigned lane_id() { return threadIdx.x & 31u; }

// 16-byte read-only streaming load: data read once, do not keep it in L1.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void st_v4(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// BF16 <-> fp32. Widening is exact (BF16 is the top half of an fp32 pattern).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Two fp32 -> packed BF16x2, round to nearest even (lo in bits 0-15).
__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two fp32 -> packed e4m3x2, round to nearest even, saturating to +-448
// (lo in bits 0-7).
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return (uint32_t)r;
}

// One e4m3 code -> its exact value (e4m3 values are exact in f16 and f32).
__device__ __forceinline__ float e4m3_to_f32(uint32_t code) {
  uint32_t h2;
  uint16_t in = (uint16_t)(code & 0xffu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
  float f;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.f32.f16 %0, lo;\n\t}"
      : "=f"(f)
      : "r"(h2));
  return f;
}

// Two fp32 -> packed e2m1x2 byte, round to nearest even, saturating to +-6
// (lo in bits 0-3, hi in bits 4-7).
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}

// Bulk asynchronous copy shared -> global (no tensor map). Both addresses
// 16-byte aligned, size a multiple of 16. Tracked in the issuing thread's
// bulk group.
__device__ __forceinline__ void bulk_store_s2g(void* gdst, const void* ssrc, uint32_t bytes) {
  uint32_t sa = (uint32_t)__cvta_generic_to_shared(ssrc);
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(sa),
               "r"(bytes)
               : "memory");
}
// Same, with an L2 evict-first policy: data written once and not read again
// soon leaves L2 early instead of staying dirty for later kernels to write
// back.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void bulk_store_s2g_evict_first(void* gdst, const void* ssrc,
                                                           uint32_t bytes, uint64_t pol) {
  uint32_t sa = (uint32_t)__cvta_generic_to_shared(ssrc);
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(gdst),
               "r"(sa), "r"(bytes), "l"(pol)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until the issuing thread's bulk copies have finished reading shared
// memory (the shared buffer may then be reused or the block may exit).
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Make generic-proxy writes to shared memory visible to the async proxy.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- mbarriers and bulk copies global -> shared -----------------------------
// An mbarrier in shared memory counts thread arrivals and the bytes of bulk
// copies (transaction count) of its current phase; waiting on the phase's
// parity returns once both are complete.
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
// Makes initialised barriers visible to the bulk-copy (async) proxy.
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// One arrival that also announces `bytes` of bulk copies for this phase.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Non-blocking form: true once the phase with this parity has completed.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Every wait on an mbarrier in this library is bounded: it gives up after
// limit_ns of wall time (kWaitLimitNs unless moe_set_wait_limit_ns lowered it
// for a test; far beyond any legitimate wait: the copies it waits for are
// reads of this GPU's own memory) and returns false, and the caller records
// MOE_ERR_TIMEOUT in the library's device status word.
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns = kWaitLimitNs) {
  if (limit_ns < kWaitLimitNs) {
    // a lowered budget (test hook): poll without suspending, since try_wait
    // may sleep longer than the budget before it reports
    const uint64_t t0 = global_timer_ns();
    while (!mbar_test_wait(bar, parity)) {
      if (global_timer_ns() - t0 > limit_ns) return false;
    }
    return true;
  }
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
  return true;
}
// Bulk copy global -> shared of `bytes` (16-byte aligned addresses, a
// multiple of 16 bytes) whose completion is counted on `bar`, with an L2
// cache policy (e.g. evict-first for data read once).
__device__ __forceinline__ void bulk_g2s(void* sdst, const void* gsrc, uint32_t bytes, uint64_t* bar,
                                         uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(sdst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

// Inclusive warp scan of an int.
__device__ __forceinline__ int warp_inclusive_scan(int v) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(0xffffffffu, v, o);
    if ((int)lane_id() >= o) v += n;
  }
  return v;
}

// Exclusive prefix sum of the per-thread values v over the block (all threads
// must call). scratch holds >= 33 ints of shared memory. Returns the
// exclusive prefix; *total gets the block sum.
template <int NT>
__device__ __forceinline__ int block_exclusive_scan(int v, int* scratch, int* total) {
  constexpr int NW = NT / 32;
  const int warp = threadIdx.x >> 5;
  int inc = warp_inclusive_scan(v);
  if (lane_id() == 31) scratch[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int w = (lane_id() < NW) ? scratch[lane_id()] : 0;
    int wi = warp_inclusive_scan(w);
    if (lane_id() < NW) scratch[lane_id()] = wi - w;
    if (lane_id() == NW - 1) scratch[32] = wi;
  }
  __syncthreads();
  int ex = scratch[warp] + inc - v;
  *total = scratch[32];
  __syncthreads();
  return ex;
}

#endif  // __CUDACC__

}  // namespace moe
