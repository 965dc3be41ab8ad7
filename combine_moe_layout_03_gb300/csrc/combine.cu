// combine.cu -- combine of MoE dispatch on sm_103a.
//
// * Top-k weighted reduction of expert outputs back to token order (DeepEP
//   repository, csrc/deep_ep.cpp Buffer::low_latency_combine):
//     out[t] = bf16_rn( fp32 fma chain, ascending j, of w[t,j] * y[slot_of[t,j]] )
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
// Design: HBM-bound gathers. A block of 128 threads covers one token and
// 128 16-byte column chunks of it (grid.y walks the hidden dimension), so
// every thread owns 8 columns. A thread first issues the loads of all its
// pairs' rows (up to 8 at a time, read-only, no L1 allocation: each expert
// row is read exactly once), then runs the fp32 fma chain in the fixed
// order. No shared-memory staging: each loaded byte is used once.
#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int kCombineThreads = 128;
constexpr int kBatch = 8;  // rows in flight per thread

struct PairOrder {
  int slot[MOE_MAX_TOPK];
  float w[MOE_MAX_TOPK];
  int last[MOE_MAX_TOPK];  // 1 if this pair closes its rank group
  int n;
};

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

__global__ void __launch_bounds__(kCombineThreads) k_combine_topk(CombineParams p) {
  __shared__ PairOrder po;
  const int t = blockIdx.x;
  const int k = p.topk;
  if (threadIdx.x == 0) {
    // Valid pairs sorted by (rank, j) when grouping by rank, else by j: an
    // insertion sort of at most 32 keys. A pair closes its group when the
    // next pair has another rank (always true for the last pair).
    int key[MOE_MAX_TOPK];
    int n = 0;
    for (int j = 0; j < k; ++j) {
      const int64_t q = (int64_t)t * k + j;
      const int s = p.slot_of[q];
      if (s < 0 || (int64_t)s >= p.expert_out_rows) continue;
      const int r = p.group_by_rank ? p.topk_idx[q] / p.experts_per_rank : 0;
      const float w = p.topk_weights[q];
      int i = n++;
      while (i > 0 && key[i - 1] > r) {  // stable: equal ranks keep j order
        key[i] = key[i - 1];
        po.slot[i] = po.slot[i - 1];
        po.w[i] = po.w[i - 1];
        --i;
      }
      key[i] = r;
      po.slot[i] = s;
      po.w[i] = w;
    }
    for (int i = 0; i < n; ++i) po.last[i] = (i == n - 1) || (key[i + 1] != key[i]);
    po.n = n;
  }
  __syncthreads();

  const int chunks = p.hidden_size / 8;
  const int c = blockIdx.y * kCombineThreads + threadIdx.x;
  if (c >= chunks) return;
  const size_t row_bytes = (size_t)p.hidden_size * 2;
  const uint8_t* base = p.expert_out + (size_t)c * 16;
  const int n = po.n;

  float total[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  float part[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  for (int m0 = 0; m0 < n; m0 += kBatch) {
    uint4 v[kBatch];
#pragma unroll
    for (int b = 0; b < kBatch; ++b)
      if (m0 + b < n) v[b] = ld_stream_v4(base + (size_t)po.slot[m0 + b] * row_bytes);
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      if (m0 + b < n) {
        fma8(part, po.w[m0 + b], v[b]);
        if (po.last[m0 + b]) {
          // TOPK rounds its single chain as it is (a chain that underflows
          // to -0 stays -0); TOPK_RANKS adds each rank's partial to the
          // running total, starting from +0.
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            total[i] = p.group_by_rank ? __fadd_rn(total[i], part[i]) : part[i];
            part[i] = 0.0f;
          }
        }
      }
    }
  }
  uint4 o;
  o.x = pack_bf16x2_rn(total[0], total[1]);
  o.y = pack_bf16x2_rn(total[2], total[3]);
  o.z = pack_bf16x2_rn(total[4], total[5]);
  o.w = pack_bf16x2_rn(total[6], total[7]);
  st_v4(p.out + (size_t)t * row_bytes + (size_t)c * 16, o);
}

// Cross-rank sum: out[i] = bf16(sum_r float(P_r[i])), i over 16-byte chunks.
template <int RB>
__global__ void __launch_bounds__(256) k_combine_ranks(const uint8_t* partials, uint8_t* out,
                                                       int64_t chunks, int num_ranks) {
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

cudaError_t launch_combine_topk(const CombineParams& p, cudaStream_t s) {
  const int chunks = p.hidden_size / 8;
  dim3 grid((unsigned)p.num_tokens, (unsigned)((chunks + kCombineThreads - 1) / kCombineThreads));
  k_combine_topk<<<grid, kCombineThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_combine_ranks(const uint8_t* partials, uint8_t* out, int64_t rows,
                                 int hidden_size, int num_ranks, cudaStream_t s) {
  const int64_t chunks = rows * (hidden_size / 8);
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t blocks = (chunks + 255) / 256;
  const int64_t cap = (int64_t)sms * 8;
  if (blocks > cap) blocks = cap;
  k_combine_ranks<4><<<(unsigned)blocks, 256, 0, s>>>(partials, out, chunks, num_ranks);
  return cudaGetLastError();
}

}  // namespace moe
