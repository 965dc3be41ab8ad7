// backward.cu -- the backward of combine, for training (DeepEP repository,
// README "Example use in model training or inference prefilling":
// combine_backward is a dispatch of the gradient through the cached handle,
// dispatch_backward is a combine).
//
//  * k_combine_backward: for out[t] = sum_j w[t,j] * y[slot_of[t,j]],
//      grad_y[slot_of[t,j]] = bf16_rn(w[t,j] * g[t])     (fp32 product)
//      grad_w[t,j]          = sum_h g[t,h] * y[slot_of[t,j], h]  (fp32)
//    One block per token. Each thread owns 16-byte column chunks of the row:
//    it loads g once, issues the loads of the k expert rows' chunks before
//    any store (the caller's buffers do not overlap, but the compiler cannot
//    assume so and would not hoist the loads itself), writes the k scaled
//    rows with 16-byte stores, and keeps one fp32 dot partial per pair. The
//    partials are reduced by warp shuffles, then across warps in ascending
//    warp order, so the result does not depend on scheduling.
//  * k_gather_ranks_backward: the backward of the rank-row gather,
//      grad_recv[send_head[t, r]] = g[t] for every r with a slot.
//  The backward of dispatch (the sum of a token's k gradient rows) is the
//  TOPK combine with unit weights (combine.cu, null weights).
#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int kBwdThreads = 256;
constexpr int kBwdWarps = kBwdThreads / 32;

template <int KT, bool WITH_W>
__global__ void __launch_bounds__(kBwdThreads) k_combine_backward(CombineBwdParams p) {
  pdl_wait();
  pdl_trigger();
  __shared__ int s_slot[KT];
  __shared__ float s_w[KT];
  __shared__ float s_red[kBwdWarps][KT];
  const int t = blockIdx.x;
  const int k = p.topk;
  if (threadIdx.x < KT) {
    int s = -1;
    float w = 0.0f;
    if ((int)threadIdx.x < k) {
      const int64_t q = (int64_t)t * k + threadIdx.x;
      s = p.slot_of[q];
      w = p.topk_weights[q];
      if (s < 0 || (int64_t)s >= p.rows) s = -1;
    }
    s_slot[threadIdx.x] = s;
    s_w[threadIdx.x] = w;
  }
  __syncthreads();
  int slot[KT];
  float w[KT];
  float dot[KT];
#pragma unroll
  for (int j = 0; j < KT; ++j) {
    slot[j] = s_slot[j];
    w[j] = s_w[j];
    dot[j] = 0.0f;
  }
  const int chunks = p.hidden_size / 8;
  const size_t row_bytes = (size_t)p.hidden_size * 2;
  for (int c = threadIdx.x; c < chunks; c += kBwdThreads) {
    const size_t col = (size_t)c * 16;
    const uint4 gv = ld_stream_v4(p.grad_out + (size_t)t * row_bytes + col);
    float g[8] = {bf16_lo(gv.x), bf16_hi(gv.x), bf16_lo(gv.y), bf16_hi(gv.y),
                  bf16_lo(gv.z), bf16_hi(gv.z), bf16_lo(gv.w), bf16_hi(gv.w)};
    uint4 yv[KT];
    if (WITH_W) {
#pragma unroll
      for (int j = 0; j < KT; ++j)
        if (slot[j] >= 0) yv[j] = ld_stream_v4(p.expert_out + (size_t)slot[j] * row_bytes + col);
    }
#pragma unroll
    for (int j = 0; j < KT; ++j) {
      if (slot[j] < 0) continue;
      uint4 o;
      o.x = pack_bf16x2_rn(__fmul_rn(w[j], g[0]), __fmul_rn(w[j], g[1]));
      o.y = pack_bf16x2_rn(__fmul_rn(w[j], g[2]), __fmul_rn(w[j], g[3]));
      o.z = pack_bf16x2_rn(__fmul_rn(w[j], g[4]), __fmul_rn(w[j], g[5]));
      o.w = pack_bf16x2_rn(__fmul_rn(w[j], g[6]), __fmul_rn(w[j], g[7]));
      st_v4(p.grad_expert_out + (size_t)slot[j] * row_bytes + col, o);
      if (WITH_W) {
        const uint4 v = yv[j];
        float d = dot[j];
        d = __fmaf_rn(g[0], bf16_lo(v.x), d);
        d = __fmaf_rn(g[1], bf16_hi(v.x), d);
        d = __fmaf_rn(g[2], bf16_lo(v.y), d);
        d = __fmaf_rn(g[3], bf16_hi(v.y), d);
        d = __fmaf_rn(g[4], bf16_lo(v.z), d);
        d = __fmaf_rn(g[5], bf16_hi(v.z), d);
        d = __fmaf_rn(g[6], bf16_lo(v.w), d);
        d = __fmaf_rn(g[7], bf16_hi(v.w), d);
        dot[j] = d;
      }
    }
  }
  if (!WITH_W) return;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int j = 0; j < KT; ++j) {
    float d = dot[j];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
    if (lane == 0) s_red[warp][j] = d;
  }
  __syncthreads();
  if ((int)threadIdx.x < k) {
    float d = 0.0f;
    if (s_slot[threadIdx.x] >= 0) {
#pragma unroll
      for (int q = 0; q < kBwdWarps; ++q) d += s_red[q][threadIdx.x];
    }
    p.grad_weights[(int64_t)t * k + threadIdx.x] = d;
  }
}

constexpr int kGatherBwdThreads = 256;

__global__ void __launch_bounds__(kGatherBwdThreads) k_gather_ranks_backward(RankCombineBwdParams p) {
  pdl_wait();
  pdl_trigger();
  __shared__ int s_slot[MOE_MAX_RANKS];
  __shared__ int s_cnt[2];
  const int t = blockIdx.x;
  const int R = p.num_ranks;
  // lanes of warps 0 and 1 load send_head[t, r] together; the valid slots are
  // compacted by ballot
  int s = -1;
  bool ok = false;
  unsigned m = 0;
  if (threadIdx.x < 64) {
    const int r = threadIdx.x;
    s = r < R ? p.send_head[(int64_t)t * R + r] : -1;
    ok = s >= 0 && (int64_t)s < p.rows;
    m = __ballot_sync(0xffffffffu, ok);
    if ((r & 31) == 0) s_cnt[r >> 5] = __popc(m);
  }
  __syncthreads();
  if (threadIdx.x < 64 && ok) {
    const int r = threadIdx.x;
    s_slot[__popc(m & ((1u << (r & 31)) - 1u)) + (r >= 32 ? s_cnt[0] : 0)] = s;
  }
  __syncthreads();
  const int n = s_cnt[0] + s_cnt[1];
  const int chunks = p.hidden_size / 8;
  const size_t row_bytes = (size_t)p.hidden_size * 2;
  for (int c = threadIdx.x; c < chunks; c += kGatherBwdThreads) {
    const uint4 g = ld_stream_v4(p.grad_out + (size_t)t * row_bytes + (size_t)c * 16);
    for (int m = 0; m < n; ++m) st_v4(p.grad_recv + (size_t)s_slot[m] * row_bytes + (size_t)c * 16, g);
  }
}

template <int KT>
const void* bwd_kernel(bool with_w) {
  return with_w ? (const void*)k_combine_backward<KT, true> : (const void*)k_combine_backward<KT, false>;
}

}  // namespace

cudaError_t launch_combine_backward(const CombineBwdParams& p, cudaStream_t s) {
  const bool with_w = p.expert_out != nullptr;
  const void* fn = p.topk <= 8 ? bwd_kernel<8>(with_w)
                 : p.topk <= 16 ? bwd_kernel<16>(with_w) : bwd_kernel<32>(with_w);
  CombineBwdParams q = p;
  void* args[] = {&q};
  return launch_pdl(fn, dim3((unsigned)p.num_tokens), dim3(kBwdThreads), 0, s, args);
}

cudaError_t launch_gather_ranks_backward(const RankCombineBwdParams& p, cudaStream_t s) {
  RankCombineBwdParams q = p;
  void* args[] = {&q};
  return launch_pdl((const void*)k_gather_ranks_backward, dim3((unsigned)p.num_tokens),
                    dim3(kGatherBwdThreads), 0, s, args);
}

}  // namespace moe
