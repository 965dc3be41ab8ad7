// combine.cu -- combine of MoE dispatch on sm_103a.
//
// * Top-k weighted reduction of expert outputs back to token order (DeepEP
//   repository, csrc/deep_ep.cpp Buffer::low_latency_combine):
//     out[t] = bf16_rn( fp32 fma chain, ascending j, of w[t,j] * y[slot_of[t,j]] )
//   With no weights (w = 1) this is the backward of dispatch: the sum of a
//   token's k gradient rows.
// * The same reduction grouped by destination rank: one fp32 partial per rank,
//   partials summed in ascending rank order, one rounding (vLLM PR
//   "Eliminate staging from NCCL symmetric reduce-scatter", Implementation:
//   the top-k reduction is written straight into the buffer the
//   reduce-scatter sums).
// * The cross-rank sum of R BF16 partials (vLLM compare view
//   ds-exp-2...ds-exp-ag, moe_reduce_scatter.cu "Lamport reduce-scatter
//   kernel" phase 3: fp32 accumulation over ranks in ascending order, one
//   BF16 round-to-nearest-even).
//
// Design: HBM-bound gathers. The work is cut into units of (token, slice of
// its 16-byte column chunks); one warp owns one unit at a time and walks the
// units of a persistent grid sized to the SMs (grid-stride over units). For
// its unit the warp loads the token's k (slot, weight, expert) with lanes
// 0..k-1, orders the valid pairs by (rank, j) with warp shuffles (no block
// barrier, no serial thread), and keeps the ordered list spread across the
// lanes. Each lane then owns one 16-byte column chunk per step: it issues the
// loads of up to 8 expert rows at once (read-only, no L1 allocation: every
// expert row is read exactly once) and runs the fp32 fma chain in the fixed
// order. The next unit's pair info is fetched while the current unit
// streams, so its latency is hidden.
#include <cstdlib>
#include <atomic>
#include <mutex>

#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int kCombineWarps = 8;  // 256 threads per block
constexpr int kBatch = 8;         // expert rows in flight per lane

__device__ __forceinline__ void fma8(float* acc, float w, uint4 v) {
  acc[0] = __fmaf_rn(w, bf16_lo(v.x), acc[0]);
  acc[1] = __fmaf_rn(w, bf16_hi(v.x), acc[1]);
  acc[2] = __fmaf_rn(w, bf16_lo(v.y), acc[2]);
  acc[3] = __fmaf_rn(w, bf16_hi(v.y), acc[3]);
  acc[4] = __fmaf_rn(w, bf16_lo(v.z), acc[4]);
  acc[5] = __fmaf_rn(w, bf16_hi(v.z), acc[5]);
  acc[6] = __fmaf_rn(w, bf16_lo(v.w), acc[6]);
  acc[7] = __fmaf_rn(w, bf16_hi(v.w), acc[7]);
}

__device__ __forceinline__ uint4 pack8(const float* a) {
  uint4 o;
  o.x = pack_bf16x2_rn(a[0], a[1]);
  o.y = pack_bf16x2_rn(a[2], a[3]);
  o.z = pack_bf16x2_rn(a[4], a[5]);
  o.w = pack_bf16x2_rn(a[6], a[7]);
  return o;
}

// The valid pairs of one token, ordered by (rank, j) when GROUP (else by j),
// spread over the warp: lane m holds the m-th pair's slot and weight; bit m of
// lastmask says whether pair m closes its rank group. Lanes 0..k-1 bring the
// token's (slot, weight, expert) in j order. All lanes must call it.
struct PairList {
  int slot;
  float w;
  unsigned lastmask;
  int n;
};

template <bool GROUP>
__device__ __forceinline__ PairList order_pairs(int slot, float w, int idx, int k, int64_t rows,
                                                int experts_per_rank) {
  const int lane = (int)lane_id();
  const bool valid = lane < k && slot >= 0 && (int64_t)slot < rows;
  const unsigned vmask = __ballot_sync(0xffffffffu, valid);
  PairList out;
  out.n = __popc(vmask);
  const int key = GROUP ? (valid ? idx / experts_per_rank : 0) : 0;
  // position of this lane's pair in (key, j) order among the valid pairs
  int pos;
  if (GROUP) {
    pos = 0;
    for (int l = 0; l < k; ++l) {
      const int kl = __shfl_sync(0xffffffffu, key, l);
      pos += ((vmask >> l) & 1u) && (kl < key || (kl == key && l < lane));
    }
  } else {
    pos = __popc(vmask & ((1u << lane) - 1u));
  }
  // lane m takes the pair at position m
  int src = 0;
  for (int l = 0; l < k; ++l) {
    const int pl = __shfl_sync(0xffffffffu, pos, l);
    if (((vmask >> l) & 1u) && pl == lane) src = l;
  }
  out.slot = __shfl_sync(0xffffffffu, slot, src);
  out.w = __shfl_sync(0xffffffffu, w, src);
  out.lastmask = 0;
  if (GROUP) {
    const int o_key = __shfl_sync(0xffffffffu, key, src);
    const int next_key = __shfl_down_sync(0xffffffffu, o_key, 1);
    out.lastmask = __ballot_sync(0xffffffffu, lane < out.n && (lane == out.n - 1 || next_key != o_key));
  }
  return out;
}

// One 16-byte column chunk of a token's combine, in fp32 (before rounding):
// GROUP = false: the fma chain over the ordered pairs; GROUP = true: the sum
// of the rank groups' chains. col points at the chunk's column in row 0 of
// expert_out. All lanes must call it (on = whether this lane's chunk exists).
template <bool GROUP>
__device__ __forceinline__ void combine_chunk(const PairList& pl, const uint8_t* col,
                                              size_t row_bytes, bool on, float* res) {
  float part[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  float total[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  for (int m0 = 0; m0 < pl.n; m0 += kBatch) {
    uint4 v[kBatch];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      v[b] = make_uint4(0, 0, 0, 0);
      if (m0 + b < pl.n) {
        const int sl = __shfl_sync(0xffffffffu, pl.slot, m0 + b);
        if (on) v[b] = ld_stream_v4(col + (size_t)sl * row_bytes);
      }
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      if (m0 + b < pl.n) {
        fma8(part, __shfl_sync(0xffffffffu, pl.w, m0 + b), v[b]);
        if (GROUP && ((pl.lastmask >> (m0 + b)) & 1u)) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            total[i] = __fadd_rn(total[i], part[i]);
            part[i] = 0.0f;
          }
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) res[i] = GROUP ? total[i] : part[i];
}

// GROUP = false: out = bf16(fma chain over j ascending)            (TOPK)
// GROUP = true:  out = bf16(sum over ranks ascending of the rank's
//                fma chain over its pairs, j ascending)             (TOPK_RANKS)
template <bool GROUP>
__global__ void __launch_bounds__(kCombineWarps * 32, 3)
    k_combine_topk(CombineParams p, int units_per_token, int chunks_per_unit, int64_t num_units) {
  pdl_wait();
  pdl_trigger();
  const int lane = (int)lane_id();
  const int k = p.topk;
  const int chunks = p.hidden_size / 8;
  const size_t row_bytes = (size_t)p.hidden_size * 2;
  const int64_t stride = (int64_t)gridDim.x * kCombineWarps;
  int64_t u = (int64_t)blockIdx.x * kCombineWarps + (threadIdx.x >> 5);

  // pair info of unit uu's token in lanes 0..k-1
  int nslot = -1, nidx = 0;
  float nw = 0.0f;
  auto fetch = [&](int64_t uu) {
    nslot = -1;
    if (uu < num_units && lane < k) {
      const int64_t q = (uu / units_per_token) * k + lane;
      nslot = p.slot_of[q];
      nw = p.topk_weights ? p.topk_weights[q] : 1.0f;
      if (GROUP) nidx = p.topk_idx[q];
    }
  };
  fetch(u);

  for (; u < num_units; u += stride) {
    const int slot = nslot, idx = nidx;
    const float w = nw;
    fetch(u + stride);  // in flight while this unit streams

    const int64_t t = u / units_per_token;
    const int c0 = (int)(u % units_per_token) * chunks_per_unit;
    const int c1 = min(c0 + chunks_per_unit, chunks);

    const PairList pl = order_pairs<GROUP>(slot, w, idx, k, p.expert_out_rows, p.experts_per_rank);
    for (int cb = c0; cb < c1; cb += 32) {
      const int c = cb + lane;
      const bool on = c < c1;
      float res[8];
      combine_chunk<GROUP>(pl, p.expert_out + (size_t)c * 16, row_bytes, on, res);
      // TOPK rounds its single chain as it is (a chain that underflows to -0
      // stays -0); TOPK_RANKS rounds the sum of the rank partials.
      if (on) st_v4(p.out + (size_t)t * row_bytes + (size_t)c * 16, pack8(res));
    }
  }
}


// The same reduction with one block per token walking its whole row: whole
// rows per block keep each expert row's bytes streaming from DRAM together,
// and the low register count lets four blocks share an SM. Used when there
// are enough tokens to fill the GPU.
constexpr int kRowThreads = 256;

template <bool GROUP, int THREADS = kRowThreads>
__global__ void __launch_bounds__(THREADS) k_combine_rows(CombineParams p) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x;
  const int lane = (int)lane_id();
  const int k = p.topk;
  const int chunks = p.hidden_size / 8;
  const size_t row_bytes = (size_t)p.hidden_size * 2;
  int slot = -1, idx = 0;
  float w = 0.0f;
  if (lane < k) {
    const int64_t qq = (int64_t)t * k + lane;
    slot = p.slot_of[qq];
    w = p.topk_weights ? p.topk_weights[qq] : 1.0f;
    if (GROUP) idx = p.topk_idx[qq];
  }
  const PairList pl = order_pairs<GROUP>(slot, w, idx, k, p.expert_out_rows, p.experts_per_rank);
  for (int cb = 0; cb < chunks; cb += THREADS) {  // uniform trip count per warp
    const int c = cb + (int)threadIdx.x;
    const bool on = c < chunks;
    float res[8];
    combine_chunk<GROUP>(pl, p.expert_out + (size_t)c * 16, row_bytes, on, res);
    if (on) st_v4(p.out + (size_t)t * row_bytes + (size_t)c * 16, pack8(res));
  }
}

// Combine fused with the residual add and RMSNorm that follow it (vLLM
// compare view ds-exp-2...ds-exp-ag, moe_rs_fused.cu: reduce-scatter + residual
// + RMSNorm in one kernel). One block per token. For each 16-byte chunk of
// the row a thread forms x = (the combine of MODE in fp32, before rounding) +
// residual, writes residual_out = bf16(x) and parks x in shared memory (so
// registers stay low and several blocks share an SM, keeping loads in
// flight while a block waits at its reduction). One block reduction gives
// sum(x^2); normed = bf16((x * rsqrt(sum/H + eps)) * gamma).
constexpr int kNormThreads = 256;

template <int MODE>
__global__ void __launch_bounds__(kNormThreads) k_combine_norm(CombineNormParams q) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ float4 xsm4[];  // [chunks][2] float4 = the row's x in fp32
  float* xsm = reinterpret_cast<float*>(xsm4);
  const CombineParams& p = q.c;
  __shared__ float red[kNormThreads / 32];
  const int t = blockIdx.x;
  const int lane = (int)lane_id(), warp = threadIdx.x >> 5;
  const int k = p.topk;
  const int chunks = p.hidden_size / 8;
  const size_t row_bytes = (size_t)p.hidden_size * 2;
  constexpr bool GROUP = MODE == MOE_COMBINE_TOPK_RANKS;

  PairList pl;
  pl.n = 0;
  pl.slot = -1;
  pl.w = 0.0f;
  pl.lastmask = 0;
  if (MODE != MOE_COMBINE_RANKS) {
    int slot = -1, idx = 0;
    float w = 0.0f;
    if (lane < k) {
      const int64_t qq = (int64_t)t * k + lane;
      slot = p.slot_of[qq];
      w = p.topk_weights ? p.topk_weights[qq] : 1.0f;
      if (GROUP) idx = p.topk_idx[qq];
    }
    pl = order_pairs<GROUP>(slot, w, idx, k, p.expert_out_rows, p.experts_per_rank);
  }

  float ss = 0.0f;
  for (int cb = 0; cb < chunks; cb += kNormThreads) {  // uniform trip count per warp
    const int c = cb + (int)threadIdx.x;
    const bool on = c < chunks;
    // the residual chunk's load goes out with the expert rows' loads
    uint4 rv = make_uint4(0, 0, 0, 0);
    if (on) rv = ld_stream_v4(q.residual_in + (size_t)t * row_bytes + (size_t)c * 16);
    float x[8];
    if (MODE == MOE_COMBINE_RANKS) {
#pragma unroll
      for (int j = 0; j < 8; ++j) x[j] = 0.0f;
      const size_t rank_stride = (size_t)p.num_tokens * row_bytes;
      const uint8_t* src = p.expert_out + (size_t)t * row_bytes + (size_t)c * 16;
      for (int r0 = 0; r0 < p.num_ranks; r0 += 4) {
        uint4 v[4];
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          v[b] = make_uint4(0, 0, 0, 0);
          if (on && r0 + b < p.num_ranks) v[b] = ld_stream_v4(src + (size_t)(r0 + b) * rank_stride);
        }
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          if (r0 + b < p.num_ranks) {
            x[0] = __fadd_rn(x[0], bf16_lo(v[b].x));
            x[1] = __fadd_rn(x[1], bf16_hi(v[b].x));
            x[2] = __fadd_rn(x[2], bf16_lo(v[b].y));
            x[3] = __fadd_rn(x[3], bf16_hi(v[b].y));
            x[4] = __fadd_rn(x[4], bf16_lo(v[b].z));
            x[5] = __fadd_rn(x[5], bf16_hi(v[b].z));
            x[6] = __fadd_rn(x[6], bf16_lo(v[b].w));
            x[7] = __fadd_rn(x[7], bf16_hi(v[b].w));
          }
        }
      }
    } else {
      combine_chunk<GROUP>(pl, p.expert_out + (size_t)c * 16, row_bytes, on, x);
    }
    if (on) {
      x[0] = __fadd_rn(x[0], bf16_lo(rv.x));
      x[1] = __fadd_rn(x[1], bf16_hi(rv.x));
      x[2] = __fadd_rn(x[2], bf16_lo(rv.y));
      x[3] = __fadd_rn(x[3], bf16_hi(rv.y));
      x[4] = __fadd_rn(x[4], bf16_lo(rv.z));
      x[5] = __fadd_rn(x[5], bf16_hi(rv.z));
      x[6] = __fadd_rn(x[6], bf16_lo(rv.w));
      x[7] = __fadd_rn(x[7], bf16_hi(rv.w));
      st_v4(q.residual_out + (size_t)t * row_bytes + (size_t)c * 16, pack8(x));
#pragma unroll
      for (int j = 0; j < 8; ++j) ss = __fmaf_rn(x[j], x[j], ss);
      xsm4[2 * c] = make_float4(x[0], x[1], x[2], x[3]);
      xsm4[2 * c + 1] = make_float4(x[4], x[5], x[6], x[7]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if (lane == 0) red[warp] = ss;
  __syncthreads();
  float tot = 0.0f;
#pragma unroll
  for (int w = 0; w < kNormThreads / 32; ++w) tot += red[w];
  const float scale = rsqrtf(__fadd_rn(__fdiv_rn(tot, (float)p.hidden_size), q.eps));
  for (int c = threadIdx.x; c < chunks; c += kNormThreads) {
    const uint4 g = *reinterpret_cast<const uint4*>(q.gamma + (size_t)c * 16);
    const float gv[8] = {bf16_lo(g.x), bf16_hi(g.x), bf16_lo(g.y), bf16_hi(g.y),
                         bf16_lo(g.z), bf16_hi(g.z), bf16_lo(g.w), bf16_hi(g.w)};
    const float* x = xsm + 8 * c;
    float y[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) y[j] = __fmul_rn(__fmul_rn(x[j], scale), gv[j]);
    st_v4(q.normed_out + (size_t)t * row_bytes + (size_t)c * 16, pack8(y));
  }
}

// The same reduction with the expert rows brought into shared memory by the
// bulk-copy engine, so the bytes in flight per SM are bounded by shared
// memory, not by registers. A unit is one slice of a token's row (up to 128
// 16-byte chunks); each block owns a contiguous run of units (mostly several
// slices of one token, so the token's pair info is loaded once). Warp 0 is
// the producer: it loads the token's (slot, weight, expert), orders the
// valid pairs as order_pairs does, writes the weights and the group mask to
// the stage's header and issues one cp.async.bulk per valid pair, copying
// the pair's row slice into the stage; the stage's "full" mbarrier counts the
// bytes. The consumer warps wait on it, run the fp32 chains of combine_chunk
// from shared memory (same operations in the same order, so the result is
// the same bit for bit), store the row slice and release the stage on its
// "empty" mbarrier. kPipeStages stages are in flight per block. Two stages of
// up to 16 KB (top-8) let about six blocks share an SM: more producers
// issuing copies at once beat deeper pipelines in fewer blocks (a sweep of
// 2/4/8 stages and 2/4/8/16 consumer warps at hidden 7168 and 8192).
constexpr int kPipeConsumerWarps = 4;
constexpr int kPipeThreads = 32 * (1 + kPipeConsumerWarps);
constexpr int kPipeStages = 2;
constexpr int kPipeMaxSliceChunks = 32 * kPipeConsumerWarps;  // one chunk per consumer thread

struct PipeHeader {  // one per stage, before its row slices
  int n;             // valid pairs
  unsigned lastmask; // bit m: pair m closes its rank group
  float w[MOE_MAX_TOPK];
};
constexpr int kPipeHeaderBytes = (int)((sizeof(PipeHeader) + 127) / 128 * 128);

// Device status word of the kernels with bounded waits: MOE_ERR_TIMEOUT once a
// wait gave up (read and cleared by moe_device_status).
__device__ int g_device_status;

__device__ __forceinline__ void record_timeout() { atomicExch(&g_device_status, MOE_ERR_TIMEOUT); }

template <bool GROUP>
__global__ void __launch_bounds__(kPipeThreads)
    k_combine_pipe(CombineParams p, int slice_chunks, int slices_per_token, int64_t num_units,
                   int64_t units_per_block, int stage_bytes, uint64_t wait_ns) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(128) uint8_t pipe_smem[];
  __shared__ __align__(8) uint64_t full[kPipeStages];
  __shared__ __align__(8) uint64_t empty[kPipeStages];
  const int warp = threadIdx.x >> 5, lane = (int)lane_id();
  const int k = p.topk;
  const int chunks = p.hidden_size / 8;
  const size_t row_bytes = (size_t)p.hidden_size * 2;
  const int64_t u0 = (int64_t)blockIdx.x * units_per_block;
  const int64_t u1 = min(u0 + units_per_block, num_units);
  if (threadIdx.x == 0) {
    for (int st = 0; st < kPipeStages; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], kPipeConsumerWarps);
    }
    mbar_init_fence();
  }
  __syncthreads();
  const int slice_bytes = slice_chunks * 16;

  if (warp == 0) {  // producer
    const uint64_t pol = l2_evict_first_policy();
    // pair info of token tt in lanes 0..k-1, fetched one token ahead
    int nslot = -1, nidx = 0;
    float nw = 0.0f;
    auto fetch = [&](int64_t tt) {
      nslot = -1;
      if (lane < k && tt * slices_per_token < u1) {
        const int64_t q = tt * k + lane;
        nslot = p.slot_of[q];
        nw = p.topk_weights ? p.topk_weights[q] : 1.0f;
        if (GROUP) nidx = p.topk_idx[q];
      }
    };
    int64_t cur_t = u0 / slices_per_token;
    fetch(cur_t);
    cur_t -= 1;
    PairList pl;
    pl.n = 0;
    pl.slot = -1;
    pl.w = 0.0f;
    pl.lastmask = 0;
    int issued = 0;
    bool ok = true;
    for (int64_t u = u0; u < u1; ++u, ++issued) {
      const int st = issued % kPipeStages;
      const int64_t t = u / slices_per_token;
      const int c0 = (int)(u % slices_per_token) * slice_chunks;
      if (t != cur_t) {  // tokens come in order: the fetched info is t's
        pl = order_pairs<GROUP>(nslot, nw, nidx, k, p.expert_out_rows, p.experts_per_rank);
        cur_t = t;
        fetch(t + 1);
      }
      // (the whole warp leaves together if any lane's wait gave up)
      if (issued >= kPipeStages &&
          !__all_sync(0xffffffffu, mbar_wait(&empty[st], ((issued / kPipeStages) + 1) & 1, wait_ns))) {
        ok = false;
        break;
      }
      uint8_t* stage = pipe_smem + (size_t)st * stage_bytes;
      PipeHeader* hdr = reinterpret_cast<PipeHeader*>(stage);
      if (lane < pl.n) hdr->w[lane] = pl.w;
      if (lane == 0) {
        hdr->n = pl.n;
        hdr->lastmask = pl.lastmask;
      }
      const uint32_t bytes = (uint32_t)(min(c0 + slice_chunks, chunks) - c0) * 16u;
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(&full[st], bytes * (uint32_t)pl.n);
      __syncwarp();
      if (lane < pl.n)
        bulk_g2s(stage + kPipeHeaderBytes + (size_t)lane * slice_bytes,
                 p.expert_out + (size_t)pl.slot * row_bytes + (size_t)c0 * 16, bytes, &full[st], pol);
    }
    if (!ok && lane == 0) record_timeout();
    // No copy may land in shared memory after the block has exited, and the
    // consumers that would otherwise hold the block until the last stage has
    // landed may have given up: wait (bounded, always with the full budget)
    // for the last phase of every stage in use.
    for (int i = max(0, issued - kPipeStages); i < issued; ++i)
      mbar_wait(&full[i % kPipeStages], (i / kPipeStages) & 1);
    return;
  }

  // consumers: thread ct owns chunk ct of every slice
  const int ct = threadIdx.x - 32;
  int done = 0;
  for (int64_t u = u0; u < u1; ++u, ++done) {
    const int st = done % kPipeStages;
    if (!__all_sync(0xffffffffu, mbar_wait(&full[st], (done / kPipeStages) & 1, wait_ns))) {
      if (lane == 0) record_timeout();
      return;
    }
    const uint8_t* stage = pipe_smem + (size_t)st * stage_bytes;
    const PipeHeader* hdr = reinterpret_cast<const PipeHeader*>(stage);
    const int n = hdr->n;
    const unsigned lastmask = hdr->lastmask;
    const int64_t t = u / slices_per_token;
    const int c0 = (int)(u % slices_per_token) * slice_chunks;
    const int c = c0 + ct;
    if (ct < slice_chunks && c < chunks) {
      const uint8_t* src = stage + kPipeHeaderBytes + (size_t)ct * 16;
      float part[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      float total[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      for (int m = 0; m < n; ++m) {
        const uint4 v = *reinterpret_cast<const uint4*>(src + (size_t)m * slice_bytes);
        fma8(part, hdr->w[m], v);
        if (GROUP && ((lastmask >> m) & 1u)) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            total[i] = __fadd_rn(total[i], part[i]);
            part[i] = 0.0f;
          }
        }
      }
      st_v4(p.out + (size_t)t * row_bytes + (size_t)c * 16, pack8(GROUP ? total : part));
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
  }
}

// Cross-rank sum: out[i] = bf16(sum_r float(P_r[i])), i over 16-byte chunks.
template <int RB>
__global__ void __launch_bounds__(256) k_combine_ranks(const uint8_t* partials, uint8_t* out,
                                                       int64_t chunks, int num_ranks) {
  pdl_wait();
  pdl_trigger();
  const size_t rank_stride = (size_t)chunks * 16;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < chunks;
       i += (int64_t)gridDim.x * blockDim.x) {
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    const uint8_t* src = partials + (size_t)i * 16;
    for (int r0 = 0; r0 < num_ranks; r0 += RB) {
      uint4 v[RB];
#pragma unroll
      for (int b = 0; b < RB; ++b)
        if (r0 + b < num_ranks) v[b] = ld_stream_v4(src + (size_t)(r0 + b) * rank_stride);
#pragma unroll
      for (int b = 0; b < RB; ++b) {
        if (r0 + b < num_ranks) {
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
    st_v4(out + (size_t)i * 16, o);
  }
}

}  // namespace

namespace {

// SM count and resident blocks of each kernel, looked up once per device
// (std::call_once: safe when several host threads launch at once).
struct DeviceInfo {
  int sms = 0;
  int topk_blocks[2] = {0, 0};
  int rows128_blocks = 0;  // resident 128-thread blocks of the plain row kernel
  size_t smem_per_sm = 0;  // shared memory an SM offers its blocks
};
DeviceInfo g_info[64];
std::once_flag g_info_once[64];

const DeviceInfo* device_info() {
  int dev = 0, sms = 0;
  if (!current_device(&dev, &sms) || dev >= 64) return nullptr;
  DeviceInfo& d = g_info[dev];
  std::call_once(g_info_once[dev], [&d, sms] {
    int b0 = 0, b1 = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b0, k_combine_topk<false>, kCombineWarps * 32, 0) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b1, k_combine_topk<true>, kCombineWarps * 32, 0) != cudaSuccess) {
      cudaGetLastError();
      b0 = b1 = 1;
    }
    d.topk_blocks[0] = b0 > 0 ? b0 : 1;
    d.topk_blocks[1] = b1 > 0 ? b1 : 1;
    int b2 = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b2, k_combine_rows<false, 128>, 128, 0) != cudaSuccess) {
      cudaGetLastError();
      b2 = 0;
    }
    d.rows128_blocks = b2;
    int dev2 = 0, smem = 0;
    if (cudaGetDevice(&dev2) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev2) != cudaSuccess) {
      cudaGetLastError();
      smem = 0;
    }
    d.smem_per_sm = (size_t)smem;
    d.sms = sms;
  });
  return d.sms > 0 ? &d : nullptr;
}

}  // namespace

// The bounded waits' budget passed to each launch of the pipelined combine.
std::atomic<uint64_t> g_wait_limit_ns{kWaitLimitNs};

// Which combines take the pipelined kernel: MOE_COMBINE_PIPE unset or 1 the
// automatic choice of launch_combine_topk, 0 none, 2 all.
int pipe_policy() {
  static const int v = [] {
    const char* e = getenv("MOE_COMBINE_PIPE");
    if (!e || !*e) return 1;
    return (int)strtol(e, nullptr, 10);
  }();
  return v;
}

cudaError_t launch_combine_pipe(const CombineParams& p, const DeviceInfo* di, cudaStream_t s) {
  const int k = p.topk;
  const int chunks = p.hidden_size / 8;
  // slices of up to 128 chunks (2 KB), fewer for large k so that a stage
  // stays within 48 KB
  int slice = kPipeMaxSliceChunks;
  while (slice > 8 && (size_t)k * slice * 16 > 48 * 1024) slice /= 2;
  if (slice > chunks) slice = chunks;
  const int slices_per_token = (chunks + slice - 1) / slice;
  const int stage_bytes = (kPipeHeaderBytes + k * slice * 16 + 127) / 128 * 128;
  const size_t smem = (size_t)kPipeStages * stage_bytes;
  const void* fn = p.group_by_rank ? (const void*)k_combine_pipe<true> : (const void*)k_combine_pipe<false>;
  cudaError_t err = ensure_dynamic_smem(fn, smem);
  if (err != cudaSuccess) return err;
  // resident blocks per SM from shared memory (1 KB per block is reserved)
  int per_sm = di->smem_per_sm ? (int)(di->smem_per_sm / (smem + 1024)) : 1;
  if (per_sm < 1) per_sm = 1;
  if (per_sm > 8) per_sm = 8;
  const int64_t num_units = (int64_t)p.num_tokens * slices_per_token;
  int64_t blocks = (int64_t)di->sms * per_sm;
  if (blocks > num_units) blocks = num_units;
  const int64_t per_block = (num_units + blocks - 1) / blocks;
  blocks = (num_units + per_block - 1) / per_block;
  CombineParams q = p;
  int sc = slice, spt = slices_per_token, sb = stage_bytes;
  int64_t nu = num_units, upb = per_block;
  uint64_t wns = g_wait_limit_ns.load(std::memory_order_relaxed);
  void* args[] = {&q, &sc, &spt, &nu, &upb, &sb, &wns};
  return launch_pdl(fn, dim3((unsigned)blocks), dim3(kPipeThreads), smem, s, args);
}

cudaError_t launch_combine_topk(const CombineParams& p, cudaStream_t s) {
  const DeviceInfo* di = device_info();
  if (!di) return cudaErrorInvalidDevice;
  const int pipe = pipe_policy();
  if (pipe >= 2) return launch_combine_pipe(p, di, s);
  // The choice, from sweeps of the three kernels on GB300 (top-8, hidden
  // 7168 and 8192, 64 to 4096 tokens, one call after an L2 flush and calls
  // back to back):
  //  * one block per row once the rows' loads in flight (a 128-thread block
  //    keeps min(k, 8) 16-byte loads per thread) reach about 12 MB, enough to
  //    cover DRAM latency at full bandwidth: from 768 tokens of top-8 up;
  //  * below that, the persistent warp kernel when every unit of at most two
  //    32-chunk steps has a resident warp (one round of row loads per warp);
  //  * otherwise the pipelined kernel, whose bulk copies keep up to 32 KB per
  //    block in flight without registers (256 and 512 tokens of hidden 8192:
  //    12.3 -> 10.0 us and 17.1 -> 14.9 us back to back).
  const int chunks = p.hidden_size / 8;
  const int steps_per_token = (chunks + 31) / 32;  // warp steps of 32 chunks
  const int g = p.group_by_rank ? 1 : 0;
  const int64_t resident_warps = (int64_t)di->sms * di->topk_blocks[g] * kCombineWarps;
  const bool rows = (int64_t)p.num_tokens * min(p.topk, kBatch) >= 6144;
  const bool one_round = (int64_t)p.num_tokens * steps_per_token <= 2 * resident_warps;
  if (!rows && !one_round && pipe == 1) return launch_combine_pipe(p, di, s);
  // The rank-grouped form keeps two fp32 accumulators per element: its
  // 128-thread blocks (twice as many per SM) measured 5% faster at N=4096
  // and 11% at N=1024 than 256-thread ones.
  if (rows || (pipe == 0 && p.num_tokens >= di->sms * 3)) {
    CombineParams q = p;
    void* args[] = {&q};
    if (p.group_by_rank)
      return launch_pdl((const void*)k_combine_rows<true, 128>, dim3((unsigned)p.num_tokens), dim3(128), 0,
                        s, args);
    // The plain form takes 128-thread blocks too while that puts every row in
    // one wave (N=1024: 27.7 -> 27.0 us), else 256.
    if (p.num_tokens <= (int64_t)di->sms * di->rows128_blocks)
      return launch_pdl((const void*)k_combine_rows<false, 128>, dim3((unsigned)p.num_tokens), dim3(128), 0,
                        s, args);
    return launch_pdl((const void*)k_combine_rows<false>, dim3((unsigned)p.num_tokens), dim3(kRowThreads),
                      0, s, args);
  }
  // Units of one step when there is a resident warp for every one (each warp
  // then waits on one round of expert-row loads instead of two), else two.
  const int per_unit =
      steps_per_token < 2 || (int64_t)p.num_tokens * steps_per_token <= resident_warps ? 1 : 2;
  const int chunks_per_unit = per_unit * 32;
  const int units_per_token = (chunks + chunks_per_unit - 1) / chunks_per_unit;
  const int64_t num_units = (int64_t)p.num_tokens * units_per_token;
  int64_t blocks = (num_units + kCombineWarps - 1) / kCombineWarps;
  const int64_t cap = (int64_t)di->sms * di->topk_blocks[g];
  if (blocks > cap) blocks = cap;
  CombineParams q = p;
  int upt = units_per_token, cpu = chunks_per_unit;
  int64_t nu = num_units;
  void* args[] = {&q, &upt, &cpu, &nu};
  const void* fn = p.group_by_rank ? (const void*)k_combine_topk<true> : (const void*)k_combine_topk<false>;
  return launch_pdl(fn, dim3((unsigned)blocks), dim3(kCombineWarps * 32), 0, s, args);
}

void set_wait_limit_ns(uint64_t ns) {
  g_wait_limit_ns.store(ns == 0 || ns > kWaitLimitNs ? kWaitLimitNs : ns, std::memory_order_relaxed);
}

int read_device_status(int32_t* out, bool clear) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof(int)) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  if (clear && v != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int)) != cudaSuccess) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
  }
  *out = v;
  return MOE_OK;
}

cudaError_t launch_combine_ranks(const uint8_t* partials, uint8_t* out, int64_t rows,
                                 int hidden_size, int num_ranks, cudaStream_t s) {
  const DeviceInfo* di = device_info();
  if (!di) return cudaErrorInvalidDevice;
  const int64_t chunks = rows * (hidden_size / 8);
  int64_t blocks = (chunks + 255) / 256;
  const int64_t cap = (int64_t)di->sms * 8;
  if (blocks > cap) blocks = cap;
  const uint8_t* a0 = partials;
  uint8_t* a1 = out;
  int64_t a2 = chunks;
  int a3 = num_ranks;
  void* args[] = {&a0, &a1, &a2, &a3};
  return launch_pdl((const void*)k_combine_ranks<4>, dim3((unsigned)blocks), dim3(256), 0, s, args);
}

cudaError_t launch_combine_norm(const CombineNormParams& p, cudaStream_t s) {
  const size_t smem = (size_t)p.c.hidden_size * 4;  // the row's x in fp32
  const void* fn = p.mode == MOE_COMBINE_TOPK    ? (const void*)k_combine_norm<MOE_COMBINE_TOPK>
                   : p.mode == MOE_COMBINE_RANKS ? (const void*)k_combine_norm<MOE_COMBINE_RANKS>
                                                 : (const void*)k_combine_norm<MOE_COMBINE_TOPK_RANKS>;
  cudaError_t err = ensure_dynamic_smem(fn, smem);
  if (err != cudaSuccess) return err;
  CombineNormParams q = p;
  void* args[] = {&q};
  return launch_pdl(fn, dim3((unsigned)p.c.num_tokens), dim3(kNormThreads), smem, s, args);
}

}  // namespace moe
