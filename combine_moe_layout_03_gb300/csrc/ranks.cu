// ranks.cu -- dispatch and combine with one record per (token, destination
// rank), the shape of DeepEP's normal (intranode) dispatch/combine (DeepEP
// repository, csrc/deep_ep.cpp Buffer::intranode_dispatch: a token is sent to
// every rank r with is_token_in_rank[t, r]; send_head [N, R], recv_src_idx,
// a per-rank prefix, per-expert receive counts rounded up to expert_alignment;
// Buffer::intranode_combine sums each token's per-rank results back).
//
//  * k_rank_layout: one block per rank scans that rank's column of
//    is_token_in_rank over the tokens (block-wide exclusive scan): send_head,
//    recv_src_idx; block 0 also writes recv_offset (exclusive scan of
//    tokens_per_rank) and the aligned per-expert counts.
//  * k_dispatch_ranks: one block per token; the payload (and its FP8/NVFP4
//    quantisation) is built once in shared memory, as in k_dispatch; thread r
//    writes the record's first segment (header, the id row with local expert
//    ids or -1, the weight row with other ranks' weights zeroed) with 16-byte
//    stores and hands payload + scales to the bulk-copy engine.
//  * k_combine_gather_ranks: one block per token; out[t] = bf16(sum over r
//    ascending, send_head[t, r] >= 0, of float(recv_out[send_head[t, r]])).
#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int kRankLayoutThreads = 1024;
constexpr int kRankCombineThreads = 256;

__global__ void __launch_bounds__(kRankLayoutThreads) k_rank_layout(RankLayoutParams p) {
  pdl_wait();
  pdl_trigger();
  __shared__ int scratch[36];
  const int r = blockIdx.x;
  const int N = p.num_tokens, R = p.num_ranks;
  // this rank's first receive slot: exclusive scan of tokens_per_rank
  int base = 0;
  for (int q = 0; q < r; ++q) base += p.tokens_per_rank[q];
  // contiguous run of tokens per thread
  const int per = (N + kRankLayoutThreads - 1) / kRankLayoutThreads;
  const int t0 = min((int)threadIdx.x * per, N), t1 = min(t0 + per, N);
  int mine = 0;
  for (int t = t0; t < t1; ++t) mine += p.is_token_in_rank[(int64_t)t * R + r] ? 1 : 0;
  int total;
  int pos = block_exclusive_scan<kRankLayoutThreads>(mine, scratch, &total);
  for (int t = t0; t < t1; ++t) {
    const bool in = p.is_token_in_rank[(int64_t)t * R + r] != 0;
    const int slot = in ? base + pos : -1;
    p.send_head[(int64_t)t * R + r] = slot;
    if (in) {
      // slots come from the caller's tokens_per_rank: write only inside [0, N*R)
      if (p.recv_src_idx && slot >= 0 && (int64_t)slot < (int64_t)N * R) p.recv_src_idx[slot] = t;
      ++pos;
    }
  }
  if (r == 0) {
    // recv_offset, aligned per-expert counts, and -1 past the last slot
    int run = 0;
    if (threadIdx.x == 0) {
      for (int q = 0; q < R; ++q) {
        p.recv_offset[q] = run;
        run += p.tokens_per_rank[q];
      }
      p.recv_offset[R] = run;
    }
    for (int e = threadIdx.x; e < p.num_experts; e += blockDim.x) {
      const int c = p.tokens_per_expert[e];
      const int a = p.expert_alignment;
      p.recv_tokens_per_expert[e] = (c + a - 1) / a * a;
    }
  }
  if (p.recv_src_idx) {
    int all = 0;
    for (int q = 0; q < R; ++q) all += p.tokens_per_rank[q];
    const int64_t cap = (int64_t)N * R;
    const int64_t first = all < 0 ? 0 : all;
    for (int64_t s = first + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; s < cap;
         s += (int64_t)gridDim.x * blockDim.x)
      p.recv_src_idx[s] = -1;
  }
}

__global__ void __launch_bounds__(kRankCombineThreads) k_combine_gather_ranks(RankCombineParams p) {
  pdl_wait();
  pdl_trigger();
  __shared__ int s_slot[MOE_MAX_RANKS];
  __shared__ int s_n;
  const int t = blockIdx.x;
  const int R = p.num_ranks;
  if (threadIdx.x == 0) {
    int n = 0;
    for (int r = 0; r < R; ++r) {
      const int s = p.send_head[(int64_t)t * R + r];
      if (s >= 0 && (int64_t)s < p.rows) s_slot[n++] = s;
    }
    s_n = n;
  }
  __syncthreads();
  const int n = s_n;
  const int chunks = p.hidden_size / 8;
  const size_t row_bytes = (size_t)p.hidden_size * 2;
  for (int c = threadIdx.x; c < chunks; c += kRankCombineThreads) {
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    const uint8_t* col = p.recv_out + (size_t)c * 16;
    for (int m0 = 0; m0 < n; m0 += 8) {
      uint4 v[8];
#pragma unroll
      for (int b = 0; b < 8; ++b)
        if (m0 + b < n) v[b] = ld_stream_v4(col + (size_t)s_slot[m0 + b] * row_bytes);
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        if (m0 + b < n) {
          acc[0] = __fadd_rn(acc[0], bf16_lo(v[b].x));
          acc[1] = __fadd_rn(acc[1], bf16_hi(v[b].x));
          acc[2] = __fadd_rn(acc[2], bf16_lo(v[b].y));
          acc[3] = __fadd_rn(acc[3], bf16_hi(v[b].y));
          acc[4] = __fadd_rn(acc[4], bf16_lo(v[b].z));
          acc[5] = __fadd_rn(acc[5], bf16_hi(v[b].z));
          acc[6] = __fadd_rn(acc[6], bf16_lo(v[b].w));
          acc[7] = __fadd_rn(acc[7], bf16_hi(v[b].w));
        }
      }
    }
    uint4 o;
    o.x = pack_bf16x2_rn(acc[0], acc[1]);
    o.y = pack_bf16x2_rn(acc[2], acc[3]);
    o.z = pack_bf16x2_rn(acc[4], acc[5]);
    o.w = pack_bf16x2_rn(acc[6], acc[7]);
    st_v4(p.out + (size_t)t * row_bytes + (size_t)c * 16, o);
  }
}

}  // namespace

cudaError_t launch_rank_layout(const RankLayoutParams& p, cudaStream_t s) {
  RankLayoutParams q = p;
  void* args[] = {&q};
  return launch_pdl((const void*)k_rank_layout, dim3(p.num_ranks), dim3(kRankLayoutThreads), 0, s, args);
}

cudaError_t launch_combine_gather_ranks(const RankCombineParams& p, cudaStream_t s) {
  RankCombineParams q = p;
  void* args[] = {&q};
  return launch_pdl((const void*)k_combine_gather_ranks, dim3((unsigned)p.num_tokens),
                    dim3(kRankCombineThreads), 0, s, args);
}

}  // namespace moe

// ---------------------------------------------------------------------------
// Fixed-capacity, expert-major receive buffers (DeepEP repository,
// csrc/deep_ep.cpp Buffer::low_latency_dispatch: packed_recv_x
// [E_l, R * max_tokens, H], packed_recv_src_info, packed_recv_layout_range
// [E_l, R] int64, packed_recv_count [E_l]). Seen from one GPU the R ranks'
// buffers are [E, R * max_tokens, ...], expert-major. Expert e's received
// pairs are packed compactly in source-rank order, which is the stable slot
// order within e: position = slot_of[t, j] - expert_offset[e]. Source rank s
// owns tokens [s*T, (s+1)*T), T = N / R.
// ---------------------------------------------------------------------------
namespace moe {
namespace {

__global__ void k_ll_layout(LlLayoutParams p) {
  pdl_wait();
  pdl_trigger();
  const int64_t pairs = (int64_t)p.num_tokens * p.topk;
  const int64_t cap = p.capacity;
  const int T = p.num_tokens / p.num_ranks;
  const int64_t gsz = (int64_t)gridDim.x * blockDim.x;
  const int64_t g0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  // ll_slot_of and src_info of every pair
  for (int64_t q = g0; q < pairs; q += gsz) {
    const int s = p.slot_of[q];
    int64_t pos = -1;
    if (s >= 0) {
      const int e = p.topk_idx[q];
      const int64_t within = (int64_t)s - p.expert_offset[e];
      if (within >= 0 && within < cap) {
        pos = (int64_t)e * cap + within;
        const int t = (int)(q / p.topk);
        p.src_info[pos] = t - (t / T) * T;  // token index within its source rank
      }
    }
    p.ll_slot_of[q] = pos < (int64_t)INT32_MAX ? (int32_t)pos : -1;
  }
  // src_info past each expert's count, counts and layout ranges
  for (int64_t i = g0; i < (int64_t)p.num_experts * cap; i += gsz) {
    const int e = (int)(i / cap);
    const int64_t within = i - (int64_t)e * cap;
    const int64_t cnt = (int64_t)p.expert_offset[e + 1] - p.expert_offset[e];
    if (within >= cnt) p.src_info[i] = -1;
  }
  for (int64_t i = g0; i < (int64_t)p.num_experts * p.num_ranks; i += gsz) {
    const int e = (int)(i / p.num_ranks), src = (int)(i % p.num_ranks);
    // pairs of expert e whose token is below src*T / (src+1)*T: binary search
    // of the expert's ascending src_of_slot run
    const int lo0 = p.expert_offset[e], hi0 = p.expert_offset[e + 1];
    int64_t bounds[2];
    for (int b = 0; b < 2; ++b) {
      const int64_t key = (int64_t)(src + b) * T * p.topk;
      int lo = lo0, hi = hi0;
      while (lo < hi) {
        const int mid = lo + (hi - lo) / 2;
        if ((int64_t)p.src_of_slot[mid] < key) lo = mid + 1; else hi = mid;
      }
      bounds[b] = lo - lo0;
    }
    const int64_t begin = bounds[0] < cap ? bounds[0] : cap;
    const int64_t end = bounds[1] < cap ? bounds[1] : cap;
    p.layout_range[i] = (begin << 32) | (end - begin);
    if (src == 0) {
      const int64_t c = (int64_t)hi0 - lo0;
      p.recv_count[e] = (int32_t)(c < cap ? c : cap);
    }
  }
}

}  // namespace

cudaError_t launch_ll_layout(const LlLayoutParams& p, cudaStream_t s) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t work = (int64_t)p.num_experts * p.capacity;
  const int64_t pairs = (int64_t)p.num_tokens * p.topk;
  if (pairs > work) work = pairs;
  int64_t blocks = (work + 255) / 256;
  if (blocks > (int64_t)sms * 8) blocks = (int64_t)sms * 8;
  if (blocks < 1) blocks = 1;
  LlLayoutParams q = p;
  void* args[] = {&q};
  return launch_pdl((const void*)k_ll_layout, dim3((unsigned)blocks), dim3(256), 0, s, args);
}

}  // namespace moe
