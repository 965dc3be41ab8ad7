// layout.cu -- routing layout of MoE dispatch on sm_103a.
//
// Computes what DeepEP's Buffer::get_dispatch_layout returns (per-rank and
// per-expert counts, is_token_in_rank; DeepEP repository, csrc/deep_ep.cpp)
// plus the prefix offsets and the stable slot map of the (token, j) pairs
// that dispatch and combine use.
//
// Design (all integer work, latency- not bandwidth-bound):
//  * Pairs are cut into chunks of kLayoutTokensPerChunk tokens.
//  * k_layout_count: one block per chunk. One thread per token reads its k
//    ids, counts them into a shared-memory histogram, builds the token's rank
//    bitmask, writes its is_token_in_rank row and counts tokens per rank with
//    warp ballots. The chunk's histogram goes to the workspace.
//  * k_layout_assign: one block per chunk. Each block scans the per-chunk
//    histograms itself (redundantly, from L2), so no grid-wide barrier, atomic
//    counter or third kernel is needed. Inside the chunk, each warp owns a
//    contiguous run of pairs; per-warp histograms and a scan over warps give
//    every warp its starting slot per expert; within a warp the rank of a
//    pair among equal experts is popc(match_any mask & lanes below). Slots
//    thus follow ascending (t, j) inside every expert: deterministic, no
//    global atomics.
//  * Small inputs (N*k <= kSmallLayoutMaxPairs, e.g. decode) run all phases in
//    one block: one launch.
// Ids outside [-1, E) count as -1 and raise the status word.
#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int kCountThreads = 128;   // one thread per token of a chunk
constexpr int kAssignThreads = 256;  // 8 warps
constexpr int kSmallThreads = 512;   // 16 warps

__device__ __forceinline__ int checked_id(int e, int E, int* bad) {
  if (e < -1 || e >= E) {
    *bad = 1;
    e = -1;
  }
  return e;
}

// Copies topk_idx[p0, p1) into shared sids[0, p1 - p0) with every invalid id
// replaced by -1 (and *bad set). 16-byte loads when the start is aligned, so
// the block pays one round of memory latency for all its ids.
__device__ void stage_ids(const LayoutParams& p, int64_t p0, int64_t p1, int* sids, int* bad) {
  const int E = p.num_experts;
  const int len = (int)(p1 - p0);
  const int32_t* src = p.topk_idx + p0;
  int b = 0;
  if ((((uintptr_t)src) & 15) == 0) {
    const int nv = len / 4;
    for (int i = threadIdx.x; i < nv; i += blockDim.x) {
      int4 v = __ldcg(reinterpret_cast<const int4*>(src) + i);
      sids[4 * i + 0] = checked_id(v.x, E, &b);
      sids[4 * i + 1] = checked_id(v.y, E, &b);
      sids[4 * i + 2] = checked_id(v.z, E, &b);
      sids[4 * i + 3] = checked_id(v.w, E, &b);
    }
    for (int i = 4 * nv + threadIdx.x; i < len; i += blockDim.x) sids[i] = checked_id(src[i], E, &b);
  } else {
    for (int i = threadIdx.x; i < len; i += blockDim.x) sids[i] = checked_id(src[i], E, &b);
  }
  if (b) *bad = 1;
}

// Phase A over tokens [t0, t1) whose ids are staged in sids (token t0 first):
// expert histogram (cnt[E], shared), per-rank token counts (rcnt[R], shared)
// and the is_token_in_rank rows. Every thread of the block must call it.
__device__ void count_tokens(const LayoutParams& p, int t0, int t1, const int* sids, int* cnt,
                             int* rcnt) {
  const int k = p.topk, R = p.num_ranks, EPR = p.experts_per_rank;
  const int warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  for (int tb = t0 + warp * 32; tb < t1; tb += nwarps * 32) {
    const int t = tb + (int)lane_id();
    uint64_t mask = 0;
    if (t < t1) {
      const int* row_ids = sids + (t - t0) * k;
      for (int j = 0; j < k; ++j) {
        const int e = row_ids[j];
        if (e >= 0) {
          atomicAdd(&cnt[e], 1);
          mask |= 1ull << (e / EPR);
        }
      }
      uint8_t* row = p.is_token_in_rank + (int64_t)t * R;
      if ((R & 3) == 0 && (((uintptr_t)p.is_token_in_rank) & 3) == 0) {
        for (int r = 0; r < R; r += 4) {
          uint32_t w = (uint32_t)((mask >> r) & 1) | (uint32_t)((mask >> (r + 1)) & 1) << 8 |
                       (uint32_t)((mask >> (r + 2)) & 1) << 16 |
                       (uint32_t)((mask >> (r + 3)) & 1) << 24;
          *reinterpret_cast<uint32_t*>(row + r) = w;
        }
      } else {
        for (int r = 0; r < R; ++r) row[r] = (uint8_t)((mask >> r) & 1);
      }
    }
    for (int r = 0; r < R; ++r) {
      unsigned b = __ballot_sync(0xffffffffu, (mask >> r) & 1);
      if (lane_id() == 0 && b) atomicAdd(&rcnt[r], __popc(b));
    }
  }
}

// Phase C over pairs [p0, p1) of one block, ids staged in sids (pair p0
// first): base[e] is the first slot of the block's pairs of expert e. whist is
// [nwarps][E] shared scratch. Writes slot_of and src_of_slot. Every thread of
// the block must call it.
__device__ void assign_slots(const LayoutParams& p, int64_t p0, int64_t p1, const int* sids,
                             const int* base, int* whist) {
  const int E = p.num_experts;
  const int warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const unsigned lane = lane_id();
  const unsigned lt = (1u << lane) - 1u;
  const int len = (int)(p1 - p0);
  const int per = (len + nwarps - 1) / nwarps;
  const int w0 = per * warp;
  const int w1 = min(w0 + per, len);
  int* wh = whist + warp * E;

  for (int e = threadIdx.x; e < nwarps * E; e += blockDim.x) whist[e] = 0;
  __syncthreads();
  // pass 1: this warp's count per expert
  for (int qb = w0; qb < w1; qb += 32) {
    const int q = qb + (int)lane;
    const int e = (q < w1) ? sids[q] : -1;
    const unsigned m = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && (m & lt) == 0) wh[e] += __popc(m);
  }
  __syncthreads();
  // scan over warps per expert, offset by the block's base
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = base[e];
    for (int w = 0; w < nwarps; ++w) {
      int c = whist[w * E + e];
      whist[w * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
  // pass 2: slots
  for (int qb = w0; qb < w1; qb += 32) {
    const int q = qb + (int)lane;
    const int e = (q < w1) ? sids[q] : -1;
    const unsigned m = __match_any_sync(0xffffffffu, e);
    int slot = -1;
    if (e >= 0) slot = wh[e] + __popc(m & lt);
    __syncwarp();
    if (e >= 0 && (m & lt) == 0) wh[e] += __popc(m);
    __syncwarp();
    if (q < w1) {
      p.slot_of[p0 + q] = slot;
      if (p.src_of_slot && slot >= 0) p.src_of_slot[slot] = (int32_t)(p0 + q);
    }
  }
}

// src_of_slot[s] = -1 for s in [P, N*k), spread over the grid.
__device__ void clear_src_tail(const LayoutParams& p, int64_t P) {
  if (!p.src_of_slot) return;
  const int64_t n = (int64_t)p.num_tokens * p.topk;
  for (int64_t s = P + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; s < n;
       s += (int64_t)gridDim.x * blockDim.x)
    p.src_of_slot[s] = -1;
}

__global__ void __launch_bounds__(kCountThreads) k_layout_count(LayoutParams p) {
  extern __shared__ int smem[];
  const int E = p.num_experts, R = p.num_ranks;
  int* cnt = smem;
  int* rcnt = smem + E;
  int* flag = rcnt + R;
  int* sids = flag + 1;  // [tokens_per_chunk * k]
  for (int i = threadIdx.x; i < E + R + 1; i += blockDim.x) smem[i] = 0;
  const int c = blockIdx.x;
  const int t0 = c * p.tokens_per_chunk;
  const int t1 = min(t0 + p.tokens_per_chunk, p.num_tokens);
  __syncthreads();
  stage_ids(p, (int64_t)t0 * p.topk, (int64_t)t1 * p.topk, sids, flag);
  __syncthreads();
  count_tokens(p, t0, t1, sids, cnt, rcnt);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) p.chunk_hist[(int64_t)c * E + e] = cnt[e];
  for (int r = threadIdx.x; r < R; r += blockDim.x) p.chunk_rank[(int64_t)c * R + r] = rcnt[r];
  if (threadIdx.x == 0) p.chunk_flag[c] = *flag;
}

// Scans the per-chunk histograms: fills base[e] with the first slot of chunk
// c's pairs of expert e; block 0 also writes the global outputs. Returns P.
template <int NT>
__device__ int64_t scan_chunks(const LayoutParams& p, int c, int* base, int* scratch) {
  const int E = p.num_experts, R = p.num_ranks, C = p.num_chunks;
  // each thread owns a contiguous run of experts [e0, e0 + ept)
  const int ept = (E + NT - 1) / NT;
  const int e0 = threadIdx.x * ept;
  int tot_mine = 0;
  for (int i = 0; i < ept; ++i) {
    const int e = e0 + i;
    if (e >= E) break;
    int tot = 0, pre = 0;
    for (int c0 = 0; c0 < C; c0 += 8) {  // 8 independent loads in flight
      int v[8];
#pragma unroll
      for (int b = 0; b < 8; ++b)
        v[b] = (c0 + b < C) ? __ldcg(&p.chunk_hist[(int64_t)(c0 + b) * E + e]) : 0;
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        tot += v[b];
        pre += (c0 + b < c) ? v[b] : 0;
      }
    }
    base[e] = pre;       // within-expert prefix of this chunk, for now
    base[E + e] = tot;   // expert total
    tot_mine += tot;
  }
  int total;
  int ex = block_exclusive_scan<NT>(tot_mine, scratch, &total);
  for (int i = 0; i < ept; ++i) {
    const int e = e0 + i;
    if (e >= E) break;
    const int tot = base[E + e];
    if (blockIdx.x == 0) {
      p.tokens_per_expert[e] = tot;
      p.expert_offset[e] = ex;
      if (e % p.experts_per_rank == 0) p.rank_offset[e / p.experts_per_rank] = ex;
    }
    base[e] += ex;
    ex += tot;
  }
  if (blockIdx.x == 0) {
    if (threadIdx.x == 0) {
      p.expert_offset[E] = total;
      p.rank_offset[R] = total;
      int f = 0;
      for (int c2 = 0; c2 < C; ++c2) f |= __ldcg(&p.chunk_flag[c2]);
      *p.status = f ? MOE_ERR_DEVICE_IDS : MOE_OK;
    }
    for (int r = threadIdx.x; r < R; r += NT) {
      int s = 0;
      for (int c2 = 0; c2 < C; ++c2) s += __ldcg(&p.chunk_rank[(int64_t)c2 * R + r]);
      p.tokens_per_rank[r] = s;
    }
  }
  __syncthreads();
  return total;
}

__global__ void __launch_bounds__(kAssignThreads) k_layout_assign(LayoutParams p) {
  extern __shared__ int smem[];
  const int E = p.num_experts;
  int* scratch = smem;            // 33 (+3 pad)
  int* base = smem + 36;          // [2E]
  int* whist = base + 2 * E;      // [8][E]
  int* sids = whist + (kAssignThreads / 32) * E;  // [tokens_per_chunk * k]
  const int c = blockIdx.x;
  const int t0 = c * p.tokens_per_chunk;
  const int t1 = min(t0 + p.tokens_per_chunk, p.num_tokens);
  const int64_t p0 = (int64_t)t0 * p.topk, p1 = (int64_t)t1 * p.topk;
  int dummy = 0;
  stage_ids(p, p0, p1, sids, &dummy);  // in flight during the scan below
  const int64_t P = scan_chunks<kAssignThreads>(p, c, base, scratch);
  assign_slots(p, p0, p1, sids, base, whist);
  clear_src_tail(p, P);
}

// Everything in one block (small inputs).
__global__ void __launch_bounds__(kSmallThreads) k_layout_small(LayoutParams p) {
  extern __shared__ int smem[];
  const int E = p.num_experts, R = p.num_ranks;
  int* scratch = smem;          // 33 (+3 pad)
  int* cnt = smem + 36;         // [E]
  int* rcnt = cnt + E;          // [R]
  int* flag = rcnt + R;         // [1]
  int* base = flag + 1;         // [E]
  int* whist = base + E;        // [16][E]
  int* sids = whist + (kSmallThreads / 32) * E;  // [N * k]
  const int64_t pairs = (int64_t)p.num_tokens * p.topk;
  for (int i = threadIdx.x; i < E + R + 1; i += blockDim.x) cnt[i] = 0;
  __syncthreads();
  stage_ids(p, 0, pairs, sids, flag);
  __syncthreads();
  count_tokens(p, 0, p.num_tokens, sids, cnt, rcnt);
  __syncthreads();
  // exclusive scan of the expert counts
  const int ept = (E + kSmallThreads - 1) / kSmallThreads;
  const int e0 = threadIdx.x * ept;
  int mine = 0;
  for (int i = 0; i < ept && e0 + i < E; ++i) mine += cnt[e0 + i];
  int total;
  int ex = block_exclusive_scan<kSmallThreads>(mine, scratch, &total);
  for (int i = 0; i < ept && e0 + i < E; ++i) {
    const int e = e0 + i;
    p.tokens_per_expert[e] = cnt[e];
    p.expert_offset[e] = ex;
    if (e % p.experts_per_rank == 0) p.rank_offset[e / p.experts_per_rank] = ex;
    base[e] = ex;
    ex += cnt[e];
  }
  for (int r = threadIdx.x; r < R; r += blockDim.x) p.tokens_per_rank[r] = rcnt[r];
  if (threadIdx.x == 0) {
    p.expert_offset[E] = total;
    p.rank_offset[R] = total;
    *p.status = *flag ? MOE_ERR_DEVICE_IDS : MOE_OK;
  }
  __syncthreads();
  assign_slots(p, 0, pairs, sids, base, whist);
  clear_src_tail(p, total);
}

}  // namespace

size_t layout_workspace_bytes(int num_tokens, int num_experts, int num_ranks) {
  const size_t chunks = (size_t)((num_tokens + kLayoutTokensPerChunk - 1) / kLayoutTokensPerChunk);
  size_t b = 256;  // status word + padding
  b += chunks * (size_t)num_experts * 4;
  b += chunks * (size_t)num_ranks * 4;
  b += chunks * 4;
  return (b + 255) / 256 * 256;
}

static cudaError_t set_smem(const void* fn, size_t bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

cudaError_t launch_layout(const LayoutParams& p, cudaStream_t s) {
  const int E = p.num_experts, R = p.num_ranks;
  const int64_t pairs = (int64_t)p.num_tokens * p.topk;
  if (pairs <= kSmallLayoutMaxPairs) {
    const size_t smem = (size_t)(36 + E + R + 1 + E + (kSmallThreads / 32) * E + pairs) * 4;
    cudaError_t err = set_smem((const void*)k_layout_small, smem);
    if (err != cudaSuccess) return err;
    k_layout_small<<<1, kSmallThreads, smem, s>>>(p);
    return cudaGetLastError();
  }
  const size_t chunk_ids = (size_t)p.tokens_per_chunk * p.topk;
  const size_t smem_count = (size_t)(E + R + 1) * 4 + chunk_ids * 4;
  cudaError_t err = set_smem((const void*)k_layout_count, smem_count);
  if (err != cudaSuccess) return err;
  k_layout_count<<<p.num_chunks, kCountThreads, smem_count, s>>>(p);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const size_t smem_assign = (size_t)(36 + 2 * E + (kAssignThreads / 32) * E) * 4 + chunk_ids * 4;
  err = set_smem((const void*)k_layout_assign, smem_assign);
  if (err != cudaSuccess) return err;
  k_layout_assign<<<p.num_chunks, kAssignThreads, smem_assign, s>>>(p);
  return cudaGetLastError();
}

}  // namespace moe
