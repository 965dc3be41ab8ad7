// layout.cu -- routing layout of MoE dispatch on sm_103a.
//
// Computes what DeepEP's Buffer::get_dispatch_layout returns (per-rank and
// per-expert counts, is_token_in_rank; DeepEP repository, csrc/deep_ep.cpp)
// plus the prefix offsets and the stable slot map of the (token, j) pairs
// that dispatch and combine use.
//
// Design (all integer work, latency- not bandwidth-bound):
//  * Whenever a block's ids and histograms fit in shared memory (every
//    workload of the pages): one launch of a thread-block cluster of up to 16
//    blocks of 512 threads, about 2048 pairs each (k_layout_cluster).
//    Each block stages its run of ids in shared memory with 16-byte
//    asynchronous copies, builds its rank-mask rows and per-warp expert
//    histograms there, and pushes its expert counts into every block's
//    shared memory (distributed shared memory stores) before one hardware
//    cluster barrier; after it each block has all counts locally, so one
//    block scan gives the expert totals, offsets and its own prefix. Each
//    block then ranks its pairs: per-warp starting slots from a scan over
//    warps, and within a warp the rank of a pair among equal experts is the
//    number of lanes below it whose ids match on every bit. Slots follow
//    ascending (t, j) inside every expert: deterministic, no global atomics,
//    no workspace except the status word. slot_of and src_of_slot are both
//    written as coalesced runs.
//  * Larger inputs: k_layout_count (one block per 128-token chunk, chunk
//    histograms to the workspace), then k_layout_assign, where every block
//    scans the chunk histograms itself (redundantly, from L2), so no
//    grid-wide barrier or atomic counter is needed, and ranks its pairs as
//    above.
// Ids outside [-1, E) count as -1 and raise the status word.
#include <cooperative_groups.h>

#include <mutex>

#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int kCountThreads = 128;   // one thread per token of a chunk
constexpr int kAssignThreads = 256;  // 8 warps
constexpr int kClusterThreads = 512;   // 16 warps
constexpr int kClusterWarps = kClusterThreads / 32;
constexpr int kClusterMaxBlocks = 16;  // non-portable cluster size where supported, else 8
constexpr int kClusterPortableBlocks = 8;
constexpr int kPairsPerClusterBlock = 2048;
constexpr int kMinPairsPerClusterBlock = 256;
constexpr size_t kClusterMaxSmem = 200 * 1024;

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
// per-rank token counts (rcnt[R], shared), the is_token_in_rank rows and, if
// COUNT_EXPERTS, the expert histogram (cnt[E], shared). Every thread of the
// block must call it.
template <bool COUNT_EXPERTS>
__device__ void count_tokens(const LayoutParams& p, int t0, int t1, const int* sids,
                             const int* rank_of, int* cnt, int* rcnt) {
  const int k = p.topk, R = p.num_ranks;
  const int warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  // a token's ids as 16-byte vectors when they are aligned (4 ids a load, a
  // quarter of the bank conflicts of scalar reads at stride k), and its rank
  // by a shift when experts per rank is a power of two
  const bool vec = (k & 3) == 0 && (((uintptr_t)sids) & 15) == 0;
  const int epr = p.experts_per_rank;
  const bool pow2 = (epr & (epr - 1)) == 0;
  const int sh = 31 - __clz(epr);
  for (int tb = t0 + warp * 32; tb < t1; tb += nwarps * 32) {
    const int t = tb + (int)lane_id();
    uint64_t mask = 0;
    if (t < t1) {
      const int* row_ids = sids + (t - t0) * k;
      for (int j0 = 0; j0 < k; j0 += 8) {  // 8 independent reads at a time
        int ev[8];
        if (vec) {
          const int4 a = reinterpret_cast<const int4*>(row_ids + j0)[0];
          const int4 b = j0 + 4 < k ? reinterpret_cast<const int4*>(row_ids + j0)[1] : make_int4(-1, -1, -1, -1);
          ev[0] = a.x; ev[1] = a.y; ev[2] = a.z; ev[3] = a.w;
          ev[4] = b.x; ev[5] = b.y; ev[6] = b.z; ev[7] = b.w;
        } else {
#pragma unroll
          for (int b = 0; b < 8; ++b) ev[b] = (j0 + b < k) ? row_ids[j0 + b] : -1;
        }
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          if (ev[b] >= 0) {
            if (COUNT_EXPERTS) atomicAdd(&cnt[ev[b]], 1);
            mask |= 1ull << (pow2 ? (ev[b] >> sh) : rank_of[ev[b]]);
          }
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

// rank_of[e] = e / (E/R) for e < E, in shared memory (no division per pair).
__device__ __forceinline__ void fill_rank_of(const LayoutParams& p, int* rank_of) {
  for (int e = threadIdx.x; e < p.num_experts; e += blockDim.x) rank_of[e] = e / p.experts_per_rank;
}

// Bits for expert keys 0..E-1 plus the "no expert" key 2^nbits - 1 >= E.
__device__ __forceinline__ int key_bits(int E) { return 32 - __clz(E); }

// Phase C, part 1, over the len pairs staged in sids: each warp owns a
// contiguous run of them, counts its run per expert into whist[warp][E] and
// replaces each staged id by (rank of the pair among the run's pairs of the
// same expert, in order) << 11 | (id + 1). Every thread of the block must
// call it; ends with a barrier.
__device__ void warp_histograms(int E, int len, int* sids, int* whist, bool zero = true) {
  const int warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const unsigned lane = lane_id();
  const unsigned lt = (1u << lane) - 1u;
  const int per = (len + nwarps - 1) / nwarps;
  const int w0 = per * warp;
  const int w1 = min(w0 + per, len);
  const int nb = key_bits(E);
  const int none = (1 << nb) - 1;
  int* wh = whist + warp * E;
  if (zero) {
    for (int e = threadIdx.x; e < nwarps * E; e += blockDim.x) whist[e] = 0;
    __syncthreads();
  }
  constexpr int S = 4;  // steps of 32 pairs whose masks are built together
  for (int qb = w0; qb < w1; qb += 32 * S) {
    int e[S], key[S];
    unsigned m[S];
#pragma unroll
    for (int st = 0; st < S; ++st) {
      const int q = qb + 32 * st + (int)lane;
      e[st] = (q < w1) ? sids[q] : -1;
      key[st] = e[st] >= 0 ? e[st] : none;
      m[st] = 0xffffffffu;
    }
    for (int b = 0; b < nb; ++b) {
#pragma unroll
      for (int st = 0; st < S; ++st) {
        const unsigned bit = (key[st] >> b) & 1u;
        const unsigned v = __ballot_sync(0xffffffffu, bit);
        m[st] &= bit ? v : ~v;
      }
    }
#pragma unroll
    for (int st = 0; st < S; ++st) {  // in pair order: counts carry over
      const int q = qb + 32 * st + (int)lane;
      int rank = 0;
      if (e[st] >= 0) rank = wh[e[st]] + __popc(m[st] & lt);
      __syncwarp();
      if (e[st] >= 0 && (m[st] & lt) == 0) wh[e[st]] += __popc(m[st]);
      __syncwarp();
      if (q < w1) sids[q] = (rank << 11) | (e[st] + 1);
    }
  }
  __syncthreads();
}

// Phase C, part 2: base[e] is the first slot of the block's pairs of expert
// e; a scan over warps turns whist into each warp's first slot per expert and
// every pair's slot is that plus its rank from part 1. Writes
// slot_of[p0 + q] and src_of_slot. Every thread of the block must call it.
template <int NW>
__device__ void assign_from_histograms(const LayoutParams& p, int64_t p0, int len,
                                       const int* sids, const int* base, int* whist) {
  const int E = p.num_experts;
  const int warp = threadIdx.x >> 5;
  const unsigned lane = lane_id();
  const int per = (len + NW - 1) / NW;
  const int w0 = per * warp;
  const int w1 = min(w0 + per, len);
  const int* wh = whist + warp * E;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = base[e];
#pragma unroll
    for (int g0 = 0; g0 < NW; g0 += 8) {  // 8 loads in flight at a time
      int c[8];
#pragma unroll
      for (int w = 0; w < 8; ++w) c[w] = whist[(g0 + w) * E + e];
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        whist[(g0 + w) * E + e] = run;
        run += c[w];
      }
    }
  }
  __syncthreads();
  for (int q = w0 + (int)lane; q < w1; q += 32) {
    const int v = sids[q];
    const int e = (v & 2047) - 1;
    const int slot = e >= 0 ? wh[e] + (v >> 11) : -1;
    p.slot_of[p0 + q] = slot;
    if (p.src_of_slot && slot >= 0) p.src_of_slot[slot] = (int32_t)(p0 + q);
  }
}

__device__ void assign_slots(const LayoutParams& p, int64_t p0, int64_t p1, int* sids,
                             const int* base, int* whist) {
  warp_histograms(p.num_experts, (int)(p1 - p0), sids, whist);
  assign_from_histograms<kAssignThreads / 32>(p, p0, (int)(p1 - p0), sids, base, whist);
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
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(16) int smem[];
  const int E = p.num_experts, R = p.num_ranks;
  int* sids = smem;                              // [tokens_per_chunk * k], 16-byte aligned
  int* cnt = sids + p.tokens_per_chunk * p.topk;  // [E]
  int* rcnt = cnt + E;
  int* flag = rcnt + R;
  int* rank_of = flag + 1;  // [E]
  for (int i = threadIdx.x; i < E + R + 1; i += blockDim.x) cnt[i] = 0;
  fill_rank_of(p, rank_of);
  const int c = blockIdx.x;
  const int t0 = c * p.tokens_per_chunk;
  const int t1 = min(t0 + p.tokens_per_chunk, p.num_tokens);
  __syncthreads();
  stage_ids(p, (int64_t)t0 * p.topk, (int64_t)t1 * p.topk, sids, flag);
  __syncthreads();
  count_tokens<true>(p, t0, t1, sids, rank_of, cnt, rcnt);
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
    // per-rank token counts and the invalid-id flag over all chunks, 8
    // independent loads in flight per thread
    for (int r = threadIdx.x; r <= R; r += NT) {
      int s = 0;
      for (int c0 = 0; c0 < C; c0 += 8) {
        int v[8];
#pragma unroll
        for (int b = 0; b < 8; ++b)
          v[b] = (c0 + b < C) ? __ldcg(r < R ? &p.chunk_rank[(int64_t)(c0 + b) * R + r]
                                             : &p.chunk_flag[c0 + b])
                              : 0;
#pragma unroll
        for (int b = 0; b < 8; ++b) s = (r < R) ? s + v[b] : (s | v[b]);
      }
      if (r < R) {
        p.tokens_per_rank[r] = s;
      } else {
        p.expert_offset[E] = total;
        p.rank_offset[R] = total;
        *p.status = s ? MOE_ERR_DEVICE_IDS : MOE_OK;
      }
    }
  }
  __syncthreads();
  return total;
}

__global__ void __launch_bounds__(kAssignThreads) k_layout_assign(LayoutParams p) {
  pdl_wait();
  pdl_trigger();
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

// Exclusive prefix sums of two per-thread values over the block at once (all
// threads must call); scratch holds >= 80 ints. *ta, *tb get the block sums.
template <int NT>
__device__ __forceinline__ int2 block_exclusive_scan2(int a, int b, int* scratch, int* ta, int* tb) {
  constexpr int NW = NT / 32;
  const int warp = threadIdx.x >> 5;
  const int ia = warp_inclusive_scan(a), ib = warp_inclusive_scan(b);
  if (lane_id() == 31) {
    scratch[warp] = ia;
    scratch[40 + warp] = ib;
  }
  __syncthreads();
  if (warp == 0) {
    const int wa = (lane_id() < NW) ? scratch[lane_id()] : 0;
    const int wb = (lane_id() < NW) ? scratch[40 + lane_id()] : 0;
    const int sa = warp_inclusive_scan(wa), sb = warp_inclusive_scan(wb);
    if (lane_id() < NW) {
      scratch[lane_id()] = sa - wa;
      scratch[40 + lane_id()] = sb - wb;
    }
    if (lane_id() == NW - 1) {
      scratch[32] = sa;
      scratch[72] = sb;
    }
  }
  __syncthreads();
  *ta = scratch[32];
  *tb = scratch[72];
  return make_int2(scratch[warp] + ia - a, scratch[40 + warp] + ib - b);
}

// Rank masks of tokens [t0, t1) whose ids are staged in sids, L lanes per
// token (k % L == 0) so that few tokens still keep every warp busy; MASK is
// uint32_t when R <= 32. masks[t - t0] gets the token's mask. Each warp counts
// tokens per rank in registers (lane r % 32 holds rank r) and writes them to
// wrc[warp][R]; no shared atomics. Returns whether an id outside [-1, E) was
// seen. Every thread of the block must call it.
template <typename MASK, int L>
__device__ bool token_masks(const LayoutParams& p, int t0, int t1, const int* sids, const int* rank_of,
                            MASK* masks, int* wrc) {
  const int k = p.topk, R = p.num_ranks, E = p.num_experts;
  const int warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int lane = (int)lane_id();
  const int kk = k / L;      // ids per lane
  const int sub = lane % L;  // this lane's part of the token
  const int epr = p.experts_per_rank;
  const bool pow2 = (epr & (epr - 1)) == 0;
  const int sh = 31 - __clz(epr);
  const bool vec = (kk & 3) == 0;
  constexpr int TPW = 32 / L;  // tokens per warp step
  bool bad = false;
  int rc0 = 0, rc1 = 0;        // tokens of ranks lane and lane + 32
  for (int tb = t0 + warp * TPW; tb < t1; tb += nwarps * TPW) {
    const int t = tb + lane / L;
    MASK mask = 0;
    if (t < t1) {
      const int* ids = sids + (t - t0) * k + sub * kk;
      for (int j0 = 0; j0 < kk; j0 += 4) {
        int ev[4];
        if (vec) {
          const int4 a = *reinterpret_cast<const int4*>(ids + j0);
          ev[0] = a.x; ev[1] = a.y; ev[2] = a.z; ev[3] = a.w;
        } else {
#pragma unroll
          for (int b = 0; b < 4; ++b) ev[b] = (j0 + b < kk) ? ids[j0 + b] : -1;
        }
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const int e = ev[b];
          if ((unsigned)(e + 1) > (unsigned)E) bad = true;  // e < -1 or e >= E
          else if (e >= 0) mask |= (MASK)1 << (pow2 ? (e >> sh) : rank_of[e]);
        }
      }
    }
#pragma unroll
    for (int o = 1; o < L; o <<= 1) {  // OR over the token's lanes
      if (sizeof(MASK) == 8) {
        const unsigned long long m = (unsigned long long)mask;
        const unsigned lo = __shfl_xor_sync(0xffffffffu, (unsigned)m, o);
        const unsigned hi = __shfl_xor_sync(0xffffffffu, (unsigned)(m >> 32), o);
        mask |= (MASK)(((unsigned long long)hi << 32) | lo);
      } else {
        mask |= (MASK)__shfl_xor_sync(0xffffffffu, (unsigned)mask, o);
      }
    }
    const bool lead = sub == 0 && t < t1;
    if (lead) masks[t - t0] = mask;
    if (!lead) mask = 0;
    for (int r = 0; r < R; ++r) {
      const int n = __popc(__ballot_sync(0xffffffffu, (unsigned)(mask >> r) & 1u));
      if (r == lane) rc0 += n;
      if (r == lane + 32) rc1 += n;
    }
  }
  if (lane < R) wrc[warp * R + lane] = rc0;
  if (lane + 32 < R) wrc[warp * R + lane + 32] = rc1;
  return bad;
}

// Ranks of the len pairs staged in sids among equal experts inside each
// warp's contiguous run: whist[w * stride + e] counts the pairs of expert e in
// warp w's run (rows zeroed by the caller), and sids[q] becomes
// rank << 11 | (e + 1), or 0 for a pair without an expert. Within a 32-pair
// step a lane finds its peers by matching the bits of its id with ballots;
// the steps follow pair order, so ranks are in (t, j) order. S steps have
// their ballots interleaved (the caller picks S no larger than a warp's run
// needs: empty steps would cost their ballots too). Every thread of the
// block must call it.
template <int S>
__device__ void warp_ranks(int E, int len, int* sids, int* whist, int stride) {
  const int warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const unsigned lane = lane_id();
  const unsigned lt = (1u << lane) - 1u;
  const int per = (len + nwarps - 1) / nwarps;
  const int w0 = per * warp;
  const int w1 = min(w0 + per, len);
  const int nb = E > 1 ? 32 - __clz(E - 1) : 0;  // bits of the largest id
  int* wh = whist + warp * stride;
  for (int qb = w0; qb < w1; qb += 32 * S) {
    int e[S];
    unsigned m[S];
#pragma unroll
    for (int st = 0; st < S; ++st) {
      const int q = qb + 32 * st + (int)lane;
      int v = (q < w1) ? sids[q] : -1;
      if ((unsigned)v >= (unsigned)E) v = -1;
      e[st] = v;
      m[st] = __ballot_sync(0xffffffffu, v >= 0);
    }
    for (int b = 0; b < nb; ++b) {
#pragma unroll
      for (int st = 0; st < S; ++st) {
        const unsigned bit = ((unsigned)e[st] >> b) & 1u;
        const unsigned v = __ballot_sync(0xffffffffu, bit);
        m[st] &= bit ? v : ~v;
      }
    }
#pragma unroll
    for (int st = 0; st < S; ++st) {  // in pair order: counts carry over
      const int q = qb + 32 * st + (int)lane;
      int rank = 0;
      if (e[st] >= 0) rank = wh[e[st]] + __popc(m[st] & lt);
      __syncwarp();
      if (e[st] >= 0 && (m[st] & lt) == 0) wh[e[st]] += __popc(m[st]);
      __syncwarp();
      if (q < w1) sids[q] = e[st] >= 0 ? ((rank << 11) | (e[st] + 1)) : 0;
    }
  }
}

// The same ranks and counts as warp_ranks, with a lane's peers (the lanes of
// its 32-pair step holding the same expert) found through shared memory
// instead of ballots: every lane ORs its bit into mb[e] (the warp's row of
// masks, zero between steps), reads the complete mask back, and the lowest
// lane of the group adds the group to the count and clears the mask. The OR
// does not depend on the order of the lanes' atomics, so the result is
// deterministic; one atomic, one load and one store per pair replace a
// ballot per bit of the id, which bounds the pass by warp votes otherwise.
__device__ void warp_ranks_or(int E, int len, int* sids, int* whist, unsigned* mb, int stride) {
  const int warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const unsigned lane = lane_id();
  const unsigned lt = (1u << lane) - 1u;
  const int per = (len + nwarps - 1) / nwarps;
  const int w0 = per * warp;
  const int w1 = min(w0 + per, len);
  int* wh = whist + warp * stride;
  unsigned* m = mb + warp * stride;
  for (int q0 = w0; q0 < w1; q0 += 32) {
    const int q = q0 + (int)lane;
    int e = (q < w1) ? sids[q] : -1;
    if ((unsigned)e >= (unsigned)E) e = -1;
    if (e >= 0) atomicOr(&m[e], 1u << lane);
    __syncwarp();
    unsigned peers = 0;
    int rank = 0;
    if (e >= 0) {
      peers = m[e];
      rank = wh[e] + __popc(peers & lt);
    }
    __syncwarp();
    if (e >= 0 && (peers & lt) == 0) {  // the group's lowest lane
      wh[e] += __popc(peers);
      m[e] = 0u;
    }
    __syncwarp();
    if (q < w1) sids[q] = e >= 0 ? ((rank << 11) | (e + 1)) : 0;
  }
}

// Stores v at the address of local_addr in the shared memory of cluster
// block `rank`.
__device__ __forceinline__ void st_cluster_s32(int* local_addr, unsigned rank, int v) {
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(local_addr);
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
  asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(ra), "r"(v) : "memory");
}

// Shared memory of k_layout_cluster, in ints (MASK words rounded to ints),
// plus the per-chunk rank counts of the receive layout when it is computed.
__host__ __device__ inline size_t cluster_rank_ints(int tpb, int R) {
  return 2 * (size_t)((tpb + 31) / 32) * R + 3 * (size_t)R + 1;
}
__host__ __device__ inline size_t cluster_smem_ints(int tpb, int k, int E, int R, int G, bool inv,
                                                    size_t mask_bytes, bool peer_masks, bool ranks = false,
                                                    bool ll = false) {
  const size_t E4 = (size_t)((E + 3) & ~3);
  return (size_t)kClusterWarps * E4 * (peer_masks ? 2 : 1) + (size_t)tpb * k * (inv ? 2 : 1) +
         tpb * mask_bytes / 4 +
         (size_t)G * E + (size_t)G * (R + 1) + (size_t)kClusterWarps * R + 4 * (size_t)E + 80 +
         (ranks ? cluster_rank_ints(tpb, R) : 0) + (ll ? (size_t)E : 0);
}

// Everything in one launch: a cluster of G blocks (G <= 16), block c owning a
// contiguous run of tokens. Every block arrives at a first cluster barrier on
// entry and waits on it before its first remote store, so all blocks have
// started by then; the exchange below uses a second one.
//  1. The block copies its ids to shared memory (16-byte asynchronous copies)
//     while it clears its counters.
//  2. Token pass: each token's rank mask (kept in shared memory) and per-rank
//     token counts per warp.
//  3. Pair pass: per-warp expert counts and each pair's rank among its warp's
//     pairs of the same expert (peer masks through shared-memory atomics, or
//     ballots where the mask rows do not fit).
//  4. Per expert, each warp's first offset in the block and the block's
//     count; the block stores its counts into every cluster block's shared
//     memory (block 0 also gets the rank counts), then one cluster barrier.
//     Global stores all come after it, so the barrier's release does not wait
//     for them, and no block reads another's memory after it, so there is no
//     closing barrier.
//  5. From the counts of all blocks: expert totals and this block's prefix;
//     one block scan gives the expert offsets and, in the same pass, the
//     offsets of the block's own pairs per expert. Block 0 writes the counts
//     and offsets.
//  6. slot_of in pair order and the block's pairs in slot order in shared
//     memory (inv), then src_of_slot from inv, so both are coalesced stores
//     (without room for inv, src_of_slot is scattered from step 6).
//  7. With p.send_head set (moe_layout_ranks), the per-rank receive layout:
//     every block has received all blocks' tokens-per-rank counts in step 4,
//     which give each rank's base and this block's prefix; warp ballots over
//     32-token chunks of the rank masks give the positions inside the block.
//  8. With p.ll_slot_of set (moe_layout_ll; the plan then makes every source
//     rank's T tokens a whole number of blocks), the fixed-capacity layout:
//     step 6 writes each pair's position slot - expert_offset[e] (if inside
//     the capacity) and src_info; every block holds all blocks' expert counts,
//     so one warp per owned expert scans them over the blocks into the
//     (source rank) ranges and the receive count, and clears the expert's
//     unused positions.
// No workspace is used except the status word.
template <typename MASK, int L>
__global__ void __launch_bounds__(kClusterThreads)
    k_layout_cluster(LayoutParams p, int tokens_per_block, int use_inv, int use_or) {
  pdl_wait();
  pdl_trigger();
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  const int G = (int)cluster.num_blocks();
  const int c = (int)cluster.block_rank();
  // Remote shared memory may be written only once every block of the cluster
  // has started: arrive now, wait just before the first remote store. A
  // cluster of one block exchanges through its own shared memory and needs
  // neither cluster barrier.
  const bool multi = G > 1;
  if (multi) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  extern __shared__ __align__(16) int smem[];
  constexpr int NW = kClusterWarps;
  const int E = p.num_experts, R = p.num_ranks, k = p.topk;
  const int tpb = tokens_per_block;  // a multiple of 4: every segment below stays 16-byte aligned
  const int E4 = (E + 3) & ~3;
  int* whist = smem;                  // [NW][E4] per-warp expert counts, then offsets
  unsigned* mb = reinterpret_cast<unsigned*>(whist + NW * E4);  // [NW][E4] peer masks if use_or
  int* sids = whist + NW * E4 * (use_or ? 2 : 1);  // [tpb * k] ids, then packed ranks
  unsigned* inv = reinterpret_cast<unsigned*>(sids + tpb * k);  // [tpb * k] if use_inv
  MASK* masks = reinterpret_cast<MASK*>(sids + tpb * k * (use_inv ? 2 : 1));  // [tpb]
  int* allcnt = reinterpret_cast<int*>(masks + tpb);  // [G][E] every block's expert counts
  int* allr = allcnt + G * E;         // [G][R + 1] rank counts and invalid-id flag (block 0)
  int* wrc = allr + G * (R + 1);      // [NW][R] per-warp rank counts
  int* cnt = wrc + NW * R;            // [E] this block's expert counts
  int* loff = cnt + E;                // [E] first position of expert e among the block's pairs
  int* delta = loff + E;              // [E] slot = delta[e] + position
  int* rank_of = delta + E;           // [E]
  int* scratch = rank_of + E;         // [80]
  // [E] expert offsets (fixed-capacity layout), after the receive-layout area
  int* eoff = scratch + 80 + (p.send_head ? (int)cluster_rank_ints(tpb, R) : 0);
  __shared__ int s_bad;
  const int t0 = min(c * tpb, p.num_tokens);
  const int t1 = min(t0 + tpb, p.num_tokens);
  const int64_t p0 = (int64_t)t0 * k;
  const int len = (t1 - t0) * k;

  // 1.
  {
    const int32_t* src = p.topk_idx + p0;
    if ((((uintptr_t)src) & 15) == 0) {
      const int nv = len / 4;
      for (int i = threadIdx.x; i < nv; i += blockDim.x) {
        const uint32_t sa = (uint32_t)__cvta_generic_to_shared(sids + 4 * i);
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(src + 4 * i) : "memory");
      }
      for (int i = 4 * nv + threadIdx.x; i < len; i += blockDim.x) sids[i] = src[i];
    } else {
      for (int i = threadIdx.x; i < len; i += blockDim.x) sids[i] = src[i];
    }
  }
  for (int i = threadIdx.x; i < NW * E4 * (use_or ? 2 : 1) / 4; i += blockDim.x)
    reinterpret_cast<int4*>(whist)[i] = make_int4(0, 0, 0, 0);  // counts and peer masks
  if (threadIdx.x == 0) s_bad = 0;
  if (p.experts_per_rank & (p.experts_per_rank - 1)) fill_rank_of(p, rank_of);
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
  __syncthreads();

  // 2. (reads the ids that step 3 overwrites: barrier between them)
  if (token_masks<MASK, L>(p, t0, t1, sids, rank_of, masks, wrc)) s_bad = 1;
  __syncthreads();
  // 3.
  {
    const int per = (len + NW - 1) / NW;  // pairs in a warp's run
    if (use_or)
      warp_ranks_or(E, len, sids, whist, mb, E4);
    else if (per <= 32)
      warp_ranks<1>(E, len, sids, whist, E4);
    else if (per <= 64)
      warp_ranks<2>(E, len, sids, whist, E4);
    else
      warp_ranks<4>(E, len, sids, whist, E4);
  }
  __syncthreads();

  // 4.
  if (multi) asm volatile("barrier.cluster.wait.aligned;" ::: "memory");  // every block has started
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const int v = whist[w * E4 + e];
      whist[w * E4 + e] = run;
      run += v;
    }
    cnt[e] = run;
    if (multi) {
      for (int b = 0; b < G; ++b) st_cluster_s32(allcnt + c * E + e, (unsigned)b, run);
    } else {
      allcnt[e] = run;
    }
  }
  for (int r = threadIdx.x; r <= R; r += blockDim.x) {
    int s = 0;
    if (r < R) {
#pragma unroll
      for (int w = 0; w < NW; ++w) s += wrc[w * R + r];
    } else {
      s = s_bad;
    }
    if (multi) {
      if (p.send_head) {
        for (int b = 0; b < G; ++b) st_cluster_s32(allr + c * (R + 1) + r, (unsigned)b, s);
      } else {
        st_cluster_s32(allr + c * (R + 1) + r, 0u, s);
      }
    } else {
      allr[r] = s;
    }
  }
  if (multi)
    cluster.sync();  // every block's counts are in the shared memory of the blocks that need them
  else
    __syncthreads();

  // 5.
  const int ept = (E + kClusterThreads - 1) / kClusterThreads;  // <= 2
  const int e0 = threadIdx.x * ept;
  int tot[2] = {0, 0}, pre[2] = {0, 0}, own[2] = {0, 0};
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int e = e0 + i;
    if (i < ept && e < E) {
      for (int b = 0; b < G; ++b) {
        const int v = allcnt[b * E + e];
        tot[i] += v;
        pre[i] += (b < c) ? v : 0;
      }
      own[i] = cnt[e];
    }
  }
  int total, nvalid;
  int2 ex = block_exclusive_scan2<kClusterThreads>(tot[0] + tot[1], own[0] + own[1], scratch, &total,
                                                   &nvalid);
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int e = e0 + i;
    if (i < ept && e < E) {
      loff[e] = ex.y;
      delta[e] = ex.x + pre[i] - ex.y;
      if (p.ll_slot_of) eoff[e] = ex.x;
      if (c == 0) {
        p.tokens_per_expert[e] = tot[i];
        p.expert_offset[e] = ex.x;
        if (e % p.experts_per_rank == 0) p.rank_offset[e / p.experts_per_rank] = ex.x;
        if (p.send_head) {  // the receive layout's per-expert counts, aligned
          const int a = p.expert_alignment;
          p.recv_tokens_per_expert[e] = (tot[i] + a - 1) / a * a;
        }
      }
      ex.x += tot[i];
      ex.y += own[i];
    }
  }
  if (c == 0) {
    for (int r = threadIdx.x; r <= R; r += blockDim.x) {
      int s = 0;
      for (int b = 0; b < G; ++b) s = (r < R) ? s + allr[b * (R + 1) + r] : (s | allr[b * (R + 1) + r]);
      if (r < R) {
        p.tokens_per_rank[r] = s;
      } else {
        p.expert_offset[E] = total;
        p.rank_offset[R] = total;
        *p.status = s ? MOE_ERR_DEVICE_IDS : MOE_OK;
      }
    }
  }
  __syncthreads();  // loff and delta are final

  // 6.
  {
    const int warp = threadIdx.x >> 5;
    const int per = (len + NW - 1) / NW;
    const int w0 = per * warp;
    const int w1 = min(w0 + per, len);
    const int* wh = whist + warp * E4;
    for (int q = w0 + (int)lane_id(); q < w1; q += 32) {
      const int v = sids[q];
      const int e = (v & 2047) - 1;
      int slot = -1;
      if (e >= 0) {
        const int i = loff[e] + wh[e] + (v >> 11);
        slot = delta[e] + i;
        if (use_inv) inv[i] = (unsigned)q | ((unsigned)(e + 1) << 21);
        else if (p.src_of_slot) p.src_of_slot[slot] = (int32_t)(p0 + q);
      }
      p.slot_of[p0 + q] = slot;
      if (p.ll_slot_of) {  // fixed-capacity position, in source-rank then token order
        int32_t pos = -1;
        if (e >= 0) {
          const int within = slot - eoff[e];
          if (within < p.ll_capacity) {
            pos = (int32_t)((int64_t)e * p.ll_capacity + within);
            const int t = t0 + q / k;
            p.src_info[pos] = t % p.ll_tokens_per_rank;
          }
        }
        p.ll_slot_of[p0 + q] = pos;
      }
    }
  }
  {  // is_token_in_rank rows of the block's tokens
    uint8_t* rows = p.is_token_in_rank + (int64_t)t0 * R;
    const int nt = t1 - t0;
    if ((R & 3) == 0 && (((uintptr_t)rows) & 3) == 0) {
      const int wpr = R >> 2;
      const bool wp2 = (wpr & (wpr - 1)) == 0;
      const int ws = 31 - __clz(wpr);
      for (int i = threadIdx.x; i < nt * wpr; i += blockDim.x) {
        const int tt = wp2 ? (i >> ws) : (i / wpr);
        const MASK m = masks[tt] >> ((i - tt * wpr) * 4);
        reinterpret_cast<uint32_t*>(rows)[i] = (uint32_t)(m & 1) | (uint32_t)((m >> 1) & 1) << 8 |
                                               (uint32_t)((m >> 2) & 1) << 16 |
                                               (uint32_t)((m >> 3) & 1) << 24;
      }
    } else {
      for (int i = threadIdx.x; i < nt * R; i += blockDim.x) {
        const int tt = i / R;
        rows[i] = (uint8_t)((masks[tt] >> (i - tt * R)) & 1);
      }
    }
  }
  if (use_inv) {
    __syncthreads();
    for (int i = threadIdx.x; i < nvalid; i += blockDim.x) {
      const unsigned v = inv[i];
      const int e = (int)(v >> 21) - 1;
      p.src_of_slot[delta[e] + i] = (int32_t)(p0 + (int)(v & ((1u << 21) - 1)));
    }
  }
  clear_src_tail(p, total);

  // 7.
  if (p.send_head) {
    const int warp = threadIdx.x >> 5, lane = (int)lane_id();
    const int nt = t1 - t0;
    const int nch = (tpb + 31) / 32;
    unsigned* cbits = reinterpret_cast<unsigned*>(scratch + 80);  // [nch][R] rank-r bits of 32 tokens
    int* cpre = scratch + 80 + nch * R;  // [nch][R] the block's rank-r tokens before the chunk
    int* rtot = cpre + nch * R;          // [R] tokens on rank r over all blocks
    int* rbef = rtot + R;                // [R] ... of the blocks before this one
    int* rbase = rbef + R;               // [R] slot of the block's first token on rank r
    int* rtotal = rbase + R;             // [1] receive slots over all ranks
    for (int ch = warp; ch < nch; ch += NW) {
      const int tt = ch * 32 + lane;
      const MASK m = tt < nt ? masks[tt] : (MASK)0;
      for (int r = 0; r < R; ++r) {
        const unsigned bits = __ballot_sync(0xffffffffu, ((m >> r) & 1) != 0);
        if (lane == 0) cbits[ch * R + r] = bits;
      }
    }
    __syncthreads();
    // one warp per rank: prefix over the chunks (lanes = chunks), and the
    // rank's totals over all blocks and over the earlier ones (lanes = blocks)
    for (int r = warp; r < R; r += NW) {
      int carry = 0;
      for (int ch0 = 0; ch0 < nch; ch0 += 32) {
        const int ch = ch0 + lane;
        const int v = ch < nch ? __popc(cbits[ch * R + r]) : 0;
        const int inc = warp_inclusive_scan(v);
        if (ch < nch) cpre[ch * R + r] = carry + inc - v;
        carry += __shfl_sync(0xffffffffu, inc, 31);
      }
      const int a = lane < G ? allr[lane * (R + 1) + r] : 0;  // G <= 16
      const int tot = __reduce_add_sync(0xffffffffu, a);
      const int bef = __reduce_add_sync(0xffffffffu, lane < c ? a : 0);
      if (lane == 0) {
        rtot[r] = tot;
        rbef[r] = bef;
      }
    }
    __syncthreads();
    if (warp == 0) {  // rank bases: exclusive scan of the rank totals (R <= 64)
      const int v0 = lane < R ? rtot[lane] : 0, v1 = lane + 32 < R ? rtot[lane + 32] : 0;
      const int i0 = warp_inclusive_scan(v0), i1 = warp_inclusive_scan(v1);
      const int s0 = __shfl_sync(0xffffffffu, i0, 31);
      const int e0 = i0 - v0, e1 = s0 + i1 - v1;
      if (lane < R) {
        rbase[lane] = e0 + rbef[lane];
        if (c == 0) p.recv_offset[lane] = e0;
      }
      if (lane + 32 < R) {
        rbase[lane + 32] = e1 + rbef[lane + 32];
        if (c == 0) p.recv_offset[lane + 32] = e1;
      }
      const int total = s0 + __shfl_sync(0xffffffffu, i1, 31);
      if (lane == 0) {
        *rtotal = total;
        if (c == 0) p.recv_offset[R] = total;
      }
    }
    __syncthreads();
    // send_head rows of the block's tokens: one contiguous run, coalesced
    const bool pow2 = (R & (R - 1)) == 0;
    const int sh_r = 31 - __clz(R);
    int32_t* shd = p.send_head + (int64_t)t0 * R;
    for (int i = threadIdx.x; i < nt * R; i += blockDim.x) {
      const int tt = pow2 ? (i >> sh_r) : (i / R), r = i - tt * R;
      const unsigned w = cbits[(tt >> 5) * R + r];
      const int l = tt & 31;
      shd[i] = ((w >> l) & 1u) ? rbase[r] + cpre[(tt >> 5) * R + r] + __popc(w & ((1u << l) - 1u)) : -1;
    }
    if (p.recv_src_idx) {
      // rank by rank, so each rank's run of slots is written in order
      for (int r = 0; r < R; ++r) {
        for (int tt = threadIdx.x; tt < nt; tt += blockDim.x) {
          const unsigned w = cbits[(tt >> 5) * R + r];
          const int l = tt & 31;
          if ((w >> l) & 1u)
            p.recv_src_idx[rbase[r] + cpre[(tt >> 5) * R + r] + __popc(w & ((1u << l) - 1u))] = t0 + tt;
        }
      }
      const int64_t cap = (int64_t)p.num_tokens * R;
      for (int64_t q = (int64_t)*rtotal + (int64_t)c * blockDim.x + threadIdx.x; q < cap;
           q += (int64_t)G * blockDim.x)
        p.recv_src_idx[q] = -1;
    }
  }

  // 8.
  if (p.ll_slot_of) {
    const int warp = threadIdx.x >> 5, lane = (int)lane_id();
    const int64_t cap = p.ll_capacity;
    const int bps = p.ll_tokens_per_rank / tpb;  // blocks per source rank
    for (int e = c + warp * G; e < E; e += NW * G) {
      // lane b: expert e's pairs in blocks before b (G <= 16 lanes)
      const int v = lane < G ? allcnt[lane * E + e] : 0;
      const int inc = warp_inclusive_scan(v);
      const int total = __shfl_sync(0xffffffffu, inc, 31);
      const int excl = inc - v;
      // ranks lane and lane + 32: begin at block s * bps, end at block (s + 1) * bps
      for (int h = 0; h < 2; ++h) {
        const int sr = lane + 32 * h;
        const int bb = sr * bps, be = (sr + 1) * bps;
        const int b0 = __shfl_sync(0xffffffffu, excl, bb < G ? bb : 0);
        const int b1 = __shfl_sync(0xffffffffu, excl, be < G ? be : 0);
        if (sr < R) {
          const int64_t lo = bb < G ? b0 : total, hi = be < G ? b1 : total;
          const int64_t c0 = lo < cap ? lo : cap, c1 = hi < cap ? hi : cap;
          p.layout_range[(int64_t)e * R + sr] = (c0 << 32) | (c1 - c0);
        }
      }
      const int64_t used = total < cap ? total : cap;
      if (lane == 0) p.recv_count[e] = (int32_t)used;
      for (int64_t i = used + lane; i < cap; i += 32) p.src_info[(int64_t)e * cap + i] = -1;
    }
  }
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

static cudaError_t set_smem(const void* fn, size_t bytes) { return ensure_dynamic_smem(fn, bytes); }

// The cluster kernel's forms: 32- or 64-bit rank masks, 1, 2 or 4 lanes per
// token in the token pass.
static const void* cluster_kernel(bool wide, int lanes) {
  if (wide) {
    if (lanes == 4) return (const void*)k_layout_cluster<unsigned long long, 4>;
    if (lanes == 2) return (const void*)k_layout_cluster<unsigned long long, 2>;
    return (const void*)k_layout_cluster<unsigned long long, 1>;
  }
  if (lanes == 4) return (const void*)k_layout_cluster<uint32_t, 4>;
  if (lanes == 2) return (const void*)k_layout_cluster<uint32_t, 2>;
  return (const void*)k_layout_cluster<uint32_t, 1>;
}

// Cluster plan for a shape: blocks G, tokens per block, lanes per token in
// the token pass, whether src_of_slot goes through shared memory, and the
// dynamic shared memory. Up to 16 blocks where the device schedules a
// non-portable cluster of 16 (looked up once per device), else 8.
struct ClusterPlan {
  int blocks, tokens_per_block, lanes;
  bool wide, use_inv, use_or, ll;
  size_t smem;
};

static int g_cluster_blocks[64];
static std::once_flag g_cluster_once[64];

// Allows every form of the cluster kernel the non-portable cluster size and
// the largest shared memory it may use, then asks whether a cluster of 16
// fits; once per device.
static int max_cluster_blocks() {
  int dev = 0, sms = 0;
  if (!current_device(&dev, &sms) || dev >= 64) return kClusterPortableBlocks;
  std::call_once(g_cluster_once[dev], [dev] {
    int best = kClusterPortableBlocks;
    bool ok = true;
    for (int wide = 0; wide < 2; ++wide) {
      for (int lanes = 1; lanes <= 4; lanes *= 2) {
        const void* fn = cluster_kernel(wide != 0, lanes);
        ok = ok && cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess &&
             ensure_dynamic_smem(fn, kClusterMaxSmem) == cudaSuccess;
      }
    }
    if (ok) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(kClusterMaxBlocks);
      cfg.blockDim = dim3(kClusterThreads);
      cfg.dynamicSmemBytes = kClusterMaxSmem;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = kClusterMaxBlocks;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, cluster_kernel(false, 1), &cfg) == cudaSuccess && n >= 1)
        best = kClusterMaxBlocks;
    }
    cudaGetLastError();
    g_cluster_blocks[dev] = best;
  });
  return g_cluster_blocks[dev];
}

// ll_T > 0 (the fixed-capacity layout, T tokens per source rank): tokens per
// block become a divisor of T, so every source rank is a whole number of
// blocks; cp.ll stays false (and the plan is the plain one) if no divisor
// fits the cluster.
static ClusterPlan cluster_plan(int num_tokens, int topk, int num_experts, int num_ranks, bool want_inv,
                                int gmax, bool ranks = false, int ll_T = 0) {
  // about kPairsPerClusterBlock pairs per block, but small inputs still
  // spread over up to gmax blocks of at least kMinPairsPerClusterBlock
  const int64_t pairs = (int64_t)num_tokens * topk;
  int64_t per = pairs / gmax;
  if (per < kMinPairsPerClusterBlock) per = kMinPairsPerClusterBlock;
  if (per > kPairsPerClusterBlock) per = kPairsPerClusterBlock;
  int g = (int)((pairs + per - 1) / per);
  g = g < 1 ? 1 : (g > gmax ? gmax : g);
  int tpb = (num_tokens + g - 1) / g;
  tpb = (tpb + 3) / 4 * 4;  // 16-byte aligned id runs per block
  bool ll = false;
  if (ll_T > 0) {
    const int lo = tpb > (num_tokens + gmax - 1) / gmax ? tpb : (num_tokens + gmax - 1) / gmax;
    for (int d = lo; d <= ll_T; ++d) {
      if (ll_T % d == 0 && (d * topk) % 4 == 0) {
        tpb = d;
        g = num_tokens / d;
        ll = true;
        break;
      }
    }
  }
  ClusterPlan cp;
  cp.ll = ll;
  cp.blocks = g;
  cp.tokens_per_block = tpb;
  cp.wide = num_ranks > 32;
  // enough lanes per token that the token pass spreads over the block's warps
  cp.lanes = (topk % 4 == 0 && tpb * 4 <= kClusterThreads) ? 4
             : (topk % 2 == 0 && tpb * 2 <= kClusterThreads) ? 2 : 1;
  const size_t mb = cp.wide ? 8 : 4;
  // peer masks in shared memory when they fit, then the inverse map for
  // coalesced src_of_slot stores when that fits too
  cp.use_or = cluster_smem_ints(tpb, topk, num_experts, num_ranks, g, false, mb, true, ranks, ll) * 4 <=
              kClusterMaxSmem;
  cp.use_inv = want_inv && cluster_smem_ints(tpb, topk, num_experts, num_ranks, g, true, mb, cp.use_or, ranks,
                                             ll) * 4 <= kClusterMaxSmem;
  cp.smem = cluster_smem_ints(tpb, topk, num_experts, num_ranks, g, cp.use_inv, mb, cp.use_or, ranks, ll) * 4;
  return cp;
}

cudaError_t launch_layout(const LayoutParams& p, cudaStream_t s, bool* extra_done) {
  const int E = p.num_experts, R = p.num_ranks;
  ClusterPlan cp = cluster_plan(p.num_tokens, p.topk, E, R, p.src_of_slot != nullptr, max_cluster_blocks(),
                                p.send_head != nullptr, p.ll_slot_of ? p.ll_tokens_per_rank : 0);
  if (p.ll_slot_of && (!cp.ll || cp.smem > kClusterMaxSmem))  // the plain plan; the caller adds the kernel
    cp = cluster_plan(p.num_tokens, p.topk, E, R, p.src_of_slot != nullptr, max_cluster_blocks(),
                      p.send_head != nullptr);
  if (extra_done) *extra_done = false;
  if (cp.smem <= kClusterMaxSmem) {
    const void* fn = cluster_kernel(cp.wide, cp.lanes);
    cudaError_t err = set_smem(fn, cp.smem);
    if (err != cudaSuccess) return err;
    LayoutParams q = p;
    if (!cp.ll) q.ll_slot_of = nullptr;
    if (extra_done) *extra_done = q.send_head != nullptr || q.ll_slot_of != nullptr;
    int tpb = cp.tokens_per_block;
    int use_inv = cp.use_inv ? 1 : 0, use_or = cp.use_or ? 1 : 0;
    void* args[] = {&q, &tpb, &use_inv, &use_or};
    return launch_pdl(fn, dim3((unsigned)cp.blocks), dim3(kClusterThreads), cp.smem, s, args, (unsigned)cp.blocks);
  }
  const size_t chunk_ids = (size_t)p.tokens_per_chunk * p.topk;
  const size_t smem_count = (size_t)(2 * E + R + 1) * 4 + chunk_ids * 4;
  cudaError_t err = set_smem((const void*)k_layout_count, smem_count);
  if (err != cudaSuccess) return err;
  LayoutParams q = p;
  q.send_head = nullptr;  // the two-kernel path leaves the receive layouts to the caller
  q.ll_slot_of = nullptr;
  void* args[] = {&q};
  err = launch_pdl((const void*)k_layout_count, dim3(p.num_chunks), dim3(kCountThreads), smem_count, s,
                   args);
  if (err != cudaSuccess) return err;
  const size_t smem_assign = (size_t)(36 + 2 * E + (kAssignThreads / 32) * E) * 4 + chunk_ids * 4;
  err = set_smem((const void*)k_layout_assign, smem_assign);
  if (err != cudaSuccess) return err;
  return launch_pdl((const void*)k_layout_assign, dim3(p.num_chunks), dim3(kAssignThreads), smem_assign,
                    s, args);
}

}  // namespace moe
