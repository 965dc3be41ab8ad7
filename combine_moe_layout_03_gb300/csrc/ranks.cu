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

// acc[i] += float(bf16 element i of v), in fp32 round-to-nearest
__device__ __forceinline__ void add8(float* acc, uint4 v) {
  acc[0] = __fadd_rn(acc[0], bf16_lo(v.x));
  acc[1] = __fadd_rn(acc[1], bf16_hi(v.x));
  acc[2] = __fadd_rn(acc[2], bf16_lo(v.y));
  acc[3] = __fadd_rn(acc[3], bf16_hi(v.y));
  acc[4] = __fadd_rn(acc[4], bf16_lo(v.z));
  acc[5] = __fadd_rn(acc[5], bf16_hi(v.z));
  acc[6] = __fadd_rn(acc[6], bf16_lo(v.w));
  acc[7] = __fadd_rn(acc[7], bf16_hi(v.w));
}

__device__ __forceinline__ uint4 pack8_bf16(const float* a) {
  uint4 o;
  o.x = pack_bf16x2_rn(a[0], a[1]);
  o.y = pack_bf16x2_rn(a[2], a[3]);
  o.z = pack_bf16x2_rn(a[4], a[5]);
  o.w = pack_bf16x2_rn(a[6], a[7]);
  return o;
}

__global__ void __launch_bounds__(kRankCombineThreads) k_combine_gather_ranks(RankCombineParams p) {
  pdl_wait();
  pdl_trigger();
  __shared__ int s_slot[MOE_MAX_RANKS];
  __shared__ int s_cnt[2];
  const int t = blockIdx.x;
  const int R = p.num_ranks;
  // warps 0 and 1: lane r loads send_head[t, r] (all loads in flight at once);
  // the valid slots are compacted in ascending r, the summation order
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
    const int before = __popc(m & ((1u << (r & 31)) - 1u)) + (r >= 32 ? s_cnt[0] : 0);
    s_slot[before] = s;
  }
  __syncthreads();
  const int n = s_cnt[0] + s_cnt[1];
  const int chunks = p.hidden_size / 8;
  const size_t row_bytes = (size_t)p.hidden_size * 2;
  // two column chunks per thread and step, four rank rows per batch: eight
  // 16-byte loads in flight (a token reaches about half as many ranks as it
  // has pairs, so one chunk alone would leave the loads half as deep)
  for (int c0 = threadIdx.x; c0 < chunks; c0 += 2 * kRankCombineThreads) {
    const int c1 = c0 + kRankCombineThreads;
    const bool on1 = c1 < chunks;
    float acc0[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    float acc1[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int m0 = 0; m0 < n; m0 += 4) {
      uint4 v0[4], v1[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        if (m0 + b < n) {
          const uint8_t* rowp = p.recv_out + (size_t)s_slot[m0 + b] * row_bytes;
          v0[b] = ld_stream_v4(rowp + (size_t)c0 * 16);
          if (on1) v1[b] = ld_stream_v4(rowp + (size_t)c1 * 16);
        }
      }
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        if (m0 + b < n) {
          add8(acc0, v0[b]);
          if (on1) add8(acc1, v1[b]);
        }
      }
    }
    st_v4(p.out + (size_t)t * row_bytes + (size_t)c0 * 16, pack8_bf16(acc0));
    if (on1) st_v4(p.out + (size_t)t * row_bytes + (size_t)c1 * 16, pack8_bf16(acc1));
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

// Three independent jobs, each given its own blocks so that they run side by
// side (each is a short chain of dependent loads):
//  * pair blocks: ll_slot_of and src_info of every pair, from slot_of,
//    topk_idx and expert_offset;
//  * fill blocks: src_info = -1 at every position past its expert's count;
//  * range blocks: one warp per expert counts the expert's pairs per source
//    rank from its run of src_of_slot (pair indices in ascending order, so
//    source ranks are nondecreasing along the run). A run of up to
//    kRangeRegs * 32 slots is held in registers and counted with shared
//    memory atomics (one round trip of loads); a longer run is split by a
//    binary search per source rank, one lane per rank.
constexpr int kLlThreads = 256;
constexpr int kRangeRegs = 8;

struct LlGrid {
  int pair_blocks, fill_blocks, range_blocks;
};

__global__ void __launch_bounds__(kLlThreads) k_ll_layout(LlLayoutParams p, LlGrid g) {
  pdl_wait();
  pdl_trigger();
  __shared__ int s_cnt[kLlThreads / 32][MOE_MAX_RANKS];
  const int64_t cap = p.capacity;
  const int T = p.num_tokens / p.num_ranks;
  const int b = blockIdx.x;
  if (b < g.pair_blocks) {
    const int64_t pairs = (int64_t)p.num_tokens * p.topk;
    for (int64_t q = (int64_t)b * kLlThreads + threadIdx.x; q < pairs;
         q += (int64_t)g.pair_blocks * kLlThreads) {
      const int s = p.slot_of[q];
      const int e = p.topk_idx[q];
      int64_t pos = -1;
      if (s >= 0 && e >= 0 && e < p.num_experts) {
        const int64_t within = (int64_t)s - p.expert_offset[e];
        if (within >= 0 && within < cap) {
          pos = (int64_t)e * cap + within;
          const int t = (int)(q / p.topk);
          p.src_info[pos] = t - (t / T) * T;  // token index within its source rank
        }
      }
      p.ll_slot_of[q] = pos < (int64_t)INT32_MAX ? (int32_t)pos : -1;
    }
    return;
  }
  if (b < g.pair_blocks + g.fill_blocks) {
    const int64_t total = (int64_t)p.num_experts * cap;
    for (int64_t i = (int64_t)(b - g.pair_blocks) * kLlThreads + threadIdx.x; i < total;
         i += (int64_t)g.fill_blocks * kLlThreads) {
      const int e = (int)(i / cap);
      const int64_t cnt = (int64_t)p.expert_offset[e + 1] - p.expert_offset[e];
      if (i - (int64_t)e * cap >= cnt) p.src_info[i] = -1;
    }
    return;
  }
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const int R = p.num_ranks;
  const int64_t pairs_per_rank = (int64_t)T * p.topk;
  int* cnt = s_cnt[wib];
  const int warps = g.range_blocks * (kLlThreads / 32);
  for (int e = (b - g.pair_blocks - g.fill_blocks) * (kLlThreads / 32) + wib; e < p.num_experts;
       e += warps) {
    const int lo = p.expert_offset[e], hi = p.expert_offset[e + 1];
    const int len = hi - lo;
    int64_t begin_lo, begin_hi;  // begin of source ranks lane and lane + 32
    if (len <= kRangeRegs * 32) {
      for (int r = lane; r < R; r += 32) cnt[r] = 0;
      __syncwarp();
      int src[kRangeRegs];
#pragma unroll
      for (int c = 0; c < kRangeRegs; ++c) {
        const int i = c * 32 + lane;
        src[c] = i < len ? p.src_of_slot[lo + i] : -1;
      }
#pragma unroll
      for (int c = 0; c < kRangeRegs; ++c)
        if (src[c] >= 0) atomicAdd(&cnt[(int)(src[c] / pairs_per_rank)], 1);
      __syncwarp();
      // exclusive scan of the per-rank counts: lane r holds ranks r, r + 32
      const int c0 = lane < R ? cnt[lane] : 0;
      const int c1 = lane + 32 < R ? cnt[lane + 32] : 0;
      int inc0 = c0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, inc0, o);
        if (lane >= o) inc0 += v;
      }
      const int sum0 = __shfl_sync(0xffffffffu, inc0, 31);
      int inc1 = c1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, inc1, o);
        if (lane >= o) inc1 += v;
      }
      begin_lo = inc0 - c0;
      begin_hi = sum0 + inc1 - c1;
      __syncwarp();
    } else {
      // lower bound of source rank r's first pair index in the run
      int64_t bound[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int64_t key = (int64_t)(lane + 32 * h) * pairs_per_rank;
        int a = lo, z = hi;
        if (lane + 32 * h < R) {
          while (a < z) {
            const int mid = a + (z - a) / 2;
            if ((int64_t)p.src_of_slot[mid] < key) a = mid + 1; else z = mid;
          }
        }
        bound[h] = a - lo;
      }
      begin_lo = bound[0];
      begin_hi = bound[1];
    }
    // begin of rank r + 1 (the run's length after the last rank)
    const int64_t next_lo_shfl = __shfl_down_sync(0xffffffffu, begin_lo, 1);
    const int64_t first_hi = __shfl_sync(0xffffffffu, begin_hi, 0);
    const int64_t next_hi_shfl = __shfl_down_sync(0xffffffffu, begin_hi, 1);
    for (int h = 0; h < 2; ++h) {
      const int r = lane + 32 * h;
      if (r >= R) continue;
      const int64_t bg = h ? begin_hi : begin_lo;
      int64_t nx;
      if (r + 1 >= R) nx = len;
      else if (h == 0) nx = lane == 31 ? first_hi : next_lo_shfl;
      else nx = next_hi_shfl;
      const int64_t b0 = bg < cap ? bg : cap;
      const int64_t b1 = nx < cap ? nx : cap;
      p.layout_range[(int64_t)e * R + r] = (b0 << 32) | (b1 - b0);
    }
    if (lane == 0) p.recv_count[e] = (int32_t)(len < cap ? len : cap);
  }
}

}  // namespace

cudaError_t launch_ll_layout(const LlLayoutParams& p, cudaStream_t s) {
  int dev = 0, sms = 148;
  if (!current_device(&dev, &sms)) sms = 148;
  auto clamp = [&](int64_t blocks) {
    const int64_t cap = (int64_t)sms * 2;
    return (int)(blocks < 1 ? 1 : (blocks > cap ? cap : blocks));
  };
  LlGrid g;
  g.pair_blocks = clamp(((int64_t)p.num_tokens * p.topk + kLlThreads - 1) / kLlThreads);
  g.fill_blocks = clamp(((int64_t)p.num_experts * p.capacity + 4 * kLlThreads - 1) / (4 * kLlThreads));
  g.range_blocks = clamp((p.num_experts + kLlThreads / 32 - 1) / (kLlThreads / 32));
  LlLayoutParams q = p;
  void* args[] = {&q, &g};
  return launch_pdl((const void*)k_ll_layout,
                    dim3((unsigned)(g.pair_blocks + g.fill_blocks + g.range_blocks)), dim3(kLlThreads),
                    0, s, args);
}

}  // namespace moe
