// dispatch.cu -- permute and pack of MoE dispatch on sm_103a.
//
// One record per (token, top-k) pair, written to its slot (records grouped by
// destination rank and expert). Record format: an int4 header, the id and
// weight rows, the payload and its scales, each segment at a 16-byte
// boundary (DeepEP repository, csrc/config.hpp LowLatencyLayout message =
// int4 header + payload + scales; vLLM compare view ds-exp-2...ds-exp-ag,
// moe_allgather.cu "Host launcher": tensors at 16-byte-aligned offsets).
//
// Design: one block per token. The token's row is read once from HBM with
// 16-byte asynchronous copies (cp.async, all in flight together) into shared
// memory, quantised there (FP8 e4m3 per 128 channels: a
// half-warp per group; NVFP4 per 16: a lane pair per group) and the record
// body (everything after the 16-byte header) is assembled once in shared
// memory. Then thread j writes pair j's header with one 16-byte store and
// hands the body to the bulk-copy engine (cp.async.bulk shared -> global), so
// the k copies of the body cost no register traffic. The stores carry an L2
// evict-first policy: records are written once here and read by another
// kernel later, so they should not linger dirty in L2 for the next kernel to
// write back. The token's input is
// read once and k records are written: the kernel is write-bound.
#include <cstdlib>

#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int kDispatchThreads = 256;

// Zero [from, to) of the shared image (byte granularity; few bytes).
__device__ __forceinline__ void zero_bytes(uint8_t* img, int from, int to) {
  for (int i = from + threadIdx.x; i < to; i += blockDim.x) img[i] = 0;
}

// Asynchronous 16-byte copies of n16 vectors global -> shared (cp.async,
// L1 bypassed). All of them are in flight at once; cp_async_wait_all() waits
// for this thread's copies in hardware.
__device__ __forceinline__ void copy_g2s_async(uint8_t* dst, const uint8_t* src, int n16) {
  for (int i = threadIdx.x; i < n16; i += blockDim.x) {
    uint32_t sa = (uint32_t)__cvta_generic_to_shared(dst + 16 * i);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(src + 16 * i)
                 : "memory");
  }
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// FP8 e4m3 with one fp32 scale per 128 channels. A half-warp covers one
// group: 16 lanes x 8 BF16 values. amax -> a = max(amax, 1e-4) ->
// scale = a / 448, inv = 448 / a (IEEE divisions) -> q = e4m3(x * inv).
__device__ __forceinline__ void quant_fp8(const uint8_t* row, int H, uint8_t* pay, float* scl) {
  // row: the token's BF16 row staged in shared memory
  const int groups = H / 128;
  const int warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int half = (int)(lane_id() >> 4), li = (int)(lane_id() & 15);
  for (int gp = warp; gp * 2 < groups; gp += nwarps) {
    const int g = gp * 2 + half;
    const bool on = g < groups;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (on) v = *reinterpret_cast<const uint4*>(row + g * 256 + li * 16);
    float x[8] = {bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y),
                  bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w)};
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float a = fmaxf(amax, 1e-4f);
    const float inv = __fdiv_rn(448.0f, a);
    uint2 q;
    q.x = cvt_e4m3x2(__fmul_rn(x[0], inv), __fmul_rn(x[1], inv)) |
          cvt_e4m3x2(__fmul_rn(x[2], inv), __fmul_rn(x[3], inv)) << 16;
    q.y = cvt_e4m3x2(__fmul_rn(x[4], inv), __fmul_rn(x[5], inv)) |
          cvt_e4m3x2(__fmul_rn(x[6], inv), __fmul_rn(x[7], inv)) << 16;
    if (on) {
      *reinterpret_cast<uint2*>(pay + g * 128 + li * 8) = q;
      if (li == 0) scl[g] = __fdiv_rn(a, 448.0f);
    }
  }
}

// FP8 e4m3 with a power-of-two scale per 128 channels, kept as one UE8M0
// byte. Same half-warp layout as quant_fp8. a = max(amax, 1e-4) -> v = a / 448
// (IEEE) -> e = the least integer with 2^e >= v: v's exponent field, plus one
// unless its mantissa is zero (v lies in [2^-23, 2^120], always normal) ->
// q = e4m3(x * 2^-e), an exact scaling -> byte = e + 127.
__device__ __forceinline__ void quant_fp8_ue8m0(const uint8_t* row, int H, uint8_t* pay, uint8_t* scl) {
  const int groups = H / 128;
  const int warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int half = (int)(lane_id() >> 4), li = (int)(lane_id() & 15);
  for (int gp = warp; gp * 2 < groups; gp += nwarps) {
    const int g = gp * 2 + half;
    const bool on = g < groups;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (on) v = *reinterpret_cast<const uint4*>(row + g * 256 + li * 16);
    float x[8] = {bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y),
                  bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w)};
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const uint32_t vb = __float_as_uint(__fdiv_rn(fmaxf(amax, 1e-4f), 448.0f));
    const int e = (int)((vb >> 23) & 0xffu) - 127 + ((vb & 0x7fffffu) ? 1 : 0);
    const float inv = __uint_as_float((uint32_t)(127 - e) << 23);  // 2^-e
    uint2 q;
    q.x = cvt_e4m3x2(__fmul_rn(x[0], inv), __fmul_rn(x[1], inv)) |
          cvt_e4m3x2(__fmul_rn(x[2], inv), __fmul_rn(x[3], inv)) << 16;
    q.y = cvt_e4m3x2(__fmul_rn(x[4], inv), __fmul_rn(x[5], inv)) |
          cvt_e4m3x2(__fmul_rn(x[6], inv), __fmul_rn(x[7], inv)) << 16;
    if (on) {
      *reinterpret_cast<uint2*>(pay + g * 128 + li * 8) = q;
      if (li == 0) scl[g] = (uint8_t)(e + 127);
    }
  }
}

// NVFP4: e2m1 codes with one e4m3 scale byte per 16 channels. A lane pair
// covers one group: 2 lanes x 8 BF16 values. amax -> sc = e4m3(amax / 6) ->
// d = value(sc) -> q = d == 0 ? 0 : e2m1(x / d) (IEEE divisions). Byte i of
// the packed row holds element 2i (low nibble) and 2i+1 (high nibble).
__device__ __forceinline__ void quant_nvfp4(const uint8_t* row, int H, uint8_t* pay, uint8_t* scl) {
  // row: the token's BF16 row staged in shared memory
  const int chunks = H / 8;  // 16-byte input vectors; even since H % 16 == 0
  for (int cb = (threadIdx.x & ~31); cb < chunks; cb += blockDim.x) {
    const int c = cb + (int)lane_id();
    const bool on = c < chunks;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (on) v = *reinterpret_cast<const uint4*>(row + c * 16);
    float x[8] = {bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y),
                  bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w)};
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    const uint32_t sc = cvt_e4m3x2(__fdiv_rn(amax, 6.0f), 0.0f) & 0xffu;
    const float d = e4m3_to_f32(sc);
    uint32_t packed = 0;
    if (d != 0.0f) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        packed |= cvt_e2m1x2(__fdiv_rn(x[2 * i], d), __fdiv_rn(x[2 * i + 1], d)) << (8 * i);
    }
    if (on) {
      *reinterpret_cast<uint32_t*>(pay + c * 4) = packed;
      if ((c & 1) == 0) scl[c >> 1] = (uint8_t)sc;
    }
  }
}

// Routing layout of a small routing computed inside the dispatch kernel, so
// that a decode-sized moe_layout_dispatch is one launch. Every block reads
// all N*k ids (a few KB, from L2 after the first block) while its token row
// is still in flight, keeps them in shared memory and builds two expert
// histograms there: all pairs, and the pairs of tokens before its own. One
// block scan of the first gives the expert offsets, so pair j of token t goes
// to
//   slot = expert_offset[e] + (pairs of earlier tokens with expert e)
//          + (j' < j of token t with expert e)
// -- the stable counting sort of the layout, computed per block with no
// grid-wide exchange. Block 0 writes the expert counts and offsets and the
// status word; block b counts the tokens of ranks b, b + N, ..., one warp per
// rank over the staged ids; each block writes its token's slot_of row,
// is_token_in_rank row (one rank per lane, OR-reduced over the warp) and
// src_of_slot entries, and a share of the src_of_slot tail (-1 beyond P).
// Ids outside [-1, E) count as -1 and raise the status word, as in the
// layout kernels.
constexpr int kFusedMaxPairs = 2048;      // what the kernel can take
constexpr int kFusedDefaultPairs = 2048;  // where the host sends it by default
constexpr int kFusedPairsPerThread = kFusedMaxPairs / kDispatchThreads;
constexpr int kFusedExpertsPerThread = (MOE_MAX_EXPERTS + kDispatchThreads - 1) / kDispatchThreads;
constexpr int kFusedScratch = 48;  // block scan scratch [0, 33); [47] invalid-id flag

// shared ints before the staged ids: the two histograms and the scratch
__host__ __device__ __forceinline__ int fused_hist_ints(int E) { return 2 * E + kFusedScratch; }

__device__ void fused_layout(const LayoutParams& lp, int t, int* hist, int* s_slot, int64_t capacity) {
  constexpr int NT = kDispatchThreads;
  const int N = lp.num_tokens, k = lp.topk, E = lp.num_experts, R = lp.num_ranks;
  const int El = lp.experts_per_rank;
  const int NK = N * k;
  const int tid = threadIdx.x;
  int* hall = hist;              // [E] pairs per expert, then the expert offsets
  int* hbef = hist + E;          // [E] pairs per expert among tokens before t
  int* scratch = hbef + E;       // [kFusedScratch]
  int* sids = scratch + kFusedScratch;  // [NK] ids, invalid ones as -1

  // every id load in flight at once
  int ev[kFusedPairsPerThread];
#pragma unroll
  for (int i = 0; i < kFusedPairsPerThread; ++i) {
    const int q = tid + i * NT;
    ev[i] = q < NK ? lp.topk_idx[q] : -1;
  }
  for (int i = tid; i < 2 * E; i += NT) hist[i] = 0;
  if (tid == 0) scratch[kFusedScratch - 1] = 0;
  __syncthreads();

  bool bad = false;
  const int before = t * k;
#pragma unroll
  for (int i = 0; i < kFusedPairsPerThread; ++i) {
    const int q = tid + i * NT;
    int e = ev[i];
    if (e < -1 || e >= E) {
      bad = true;
      e = -1;
    } else if (e >= 0) {
      atomicAdd(&hall[e], 1);
      if (q < before) atomicAdd(&hbef[e], 1);
    }
    if (q < NK) sids[q] = e;
  }
  if (bad) scratch[kFusedScratch - 1] = 1;
  __syncthreads();

  // ranks b, b + N, ...: tokens with a pair on the rank, one warp each over
  // the staged ids (from the last warp down)
  {
    const int warp = tid >> 5, lane = (int)lane_id();
    const int owned_r = (int)blockIdx.x < R ? (R - (int)blockIdx.x + N - 1) / N : 0;
    for (int m = NT / 32 - 1 - warp; m < owned_r; m += NT / 32) {
      const int r = blockIdx.x + m * N;
      const int lo = r * El, hi = lo + El;
      int cnt = 0;
      for (int u = lane; u < N; u += 32) {
        bool hit = false;
        for (int j = 0; j < k; ++j) {
          const int x = sids[u * k + j];
          hit |= x >= lo && x < hi;
        }
        cnt += hit ? 1 : 0;
      }
      cnt = __reduce_add_sync(0xffffffffu, cnt);
      if (lane == 0) lp.tokens_per_rank[r] = cnt;
    }
  }

  // expert offsets: thread tid owns experts [tid*m, tid*m + m)
  const int m = (E + NT - 1) / NT;
  int c[kFusedExpertsPerThread];
  int sum = 0;
#pragma unroll
  for (int i = 0; i < kFusedExpertsPerThread; ++i) {
    const int e = tid * m + i;
    c[i] = (i < m && e < E) ? hall[e] : 0;
    sum += c[i];
  }
  int P = 0;
  int ex = block_exclusive_scan<NT>(sum, scratch, &P);  // ends with a barrier
  const bool lead = blockIdx.x == 0;
#pragma unroll
  for (int i = 0; i < kFusedExpertsPerThread; ++i) {
    const int e = tid * m + i;
    if (i < m && e < E) {
      if (lead) {
        lp.tokens_per_expert[e] = c[i];
        lp.expert_offset[e] = ex;
        if (e % El == 0) lp.rank_offset[e / El] = ex;
      }
      hall[e] = ex;
      ex += c[i];
    }
  }
  if (lead && tid == 0) {
    lp.expert_offset[E] = P;
    lp.rank_offset[R] = P;
    *lp.status = scratch[kFusedScratch - 1] ? MOE_ERR_DEVICE_IDS : MOE_OK;
  }
  __syncthreads();

  if (tid < k) {
    const int j = tid;
    const int e = sids[t * k + j];
    int s = -1;
    if (e >= 0) {
      s = hall[e] + hbef[e];
      for (int jj = 0; jj < j; ++jj) s += sids[t * k + jj] == e;
    }
    lp.slot_of[(int64_t)t * k + j] = s;
    if (lp.src_of_slot && s >= 0) lp.src_of_slot[s] = t * k + j;
    s_slot[j] = (s >= 0 && (int64_t)s < capacity) ? s : -1;
  }
  if (tid < 32) {  // the token's rank row: one division per lane, OR over the warp
    const int e = tid < k ? sids[t * k + tid] : -1;
    const int r = e >= 0 ? e / El : -1;
    const unsigned m0 = __reduce_or_sync(0xffffffffu, (r >= 0 && r < 32) ? 1u << r : 0u);
    const unsigned m1 = __reduce_or_sync(0xffffffffu, r >= 32 ? 1u << (r - 32) : 0u);
    for (int rr = tid; rr < R; rr += 32)
      lp.is_token_in_rank[(int64_t)t * R + rr] = (uint8_t)(((rr < 32 ? m0 >> rr : m1 >> (rr - 32))) & 1u);
  }
  if (lp.src_of_slot)
    for (int s = P + blockIdx.x * NT + tid; s < NK; s += gridDim.x * NT) lp.src_of_slot[s] = -1;
}

// How a dispatch block learns its slots:
//  kSlotsAfterWait  read slot_of after griddepcontrol.wait (moe_dispatch);
//  kSlotsEarly      only right after this library's own layout kernel (in
//                   moe_layout_dispatch): the row copy, its quantisation and
//                   the id and weight rows -- inputs the layout kernel does
//                   not write -- happen before griddepcontrol.wait,
//                   overlapping the layout; only slot_of, the layout's
//                   output, is read after it;
//  kSlotsFused      computed in the block (fused_layout) while the row copy
//                   is in flight (moe_layout_dispatch of a small routing).
constexpr int kSlotsAfterWait = 0, kSlotsEarly = 1, kSlotsFused = 2;

template <int OUT_KIND, int SLOTS>
__device__ __forceinline__ void dispatch_token(const DispatchParams& p, const LayoutParams* lp) {
  if (SLOTS != kSlotsEarly) {
    pdl_wait();
    pdl_trigger();
  }
  // Dynamic shared memory: the record body (record bytes [16, record_bytes)),
  // then, for the quantising kinds, the staged BF16 input row, then (fused
  // layout) the histograms.
  extern __shared__ __align__(128) uint8_t img[];
  __shared__ int s_slot[MOE_MAX_TOPK];
  __shared__ int s_expert[MOE_MAX_TOPK];
  const int t = blockIdx.x;
  const int k = p.topk;
  const int body = p.record_bytes - 16;
  const int oi = p.off_ids - 16, ow = p.off_weights - 16, op = p.off_payload - 16,
            os = p.off_scales - 16;
  constexpr bool kQuant = OUT_KIND == MOE_PAYLOAD_FP8_E4M3_B128 || OUT_KIND == MOE_PAYLOAD_NVFP4_B16 ||
                          OUT_KIND == MOE_PAYLOAD_FP8_E4M3_UE8M0;
  uint8_t* stage = img + body;

  // start the row's copies first so they overlap the small loads below
  const uint8_t* row = p.hidden + (size_t)t * p.in_row_bytes;
  if (kQuant) {
    copy_g2s_async(stage, row, p.in_row_bytes / 16);
  } else {
    copy_g2s_async(img + op, row, p.payload_bytes / 16);
    if (OUT_KIND == MOE_PAYLOAD_RAW && p.scale_bytes > 0)
      copy_g2s_async(img + os, p.scales + (size_t)t * p.in_scale_bytes, p.scale_bytes / 16);
  }

  // slots, ids and weights of this token (the fused form keeps the loads in
  // flight through its layout and stores them after it)
  int own_e = -1;
  uint32_t own_w = 0;
  if (threadIdx.x < k) {
    const int64_t q = (int64_t)t * k + threadIdx.x;
    if (SLOTS == kSlotsAfterWait) {
      const int s = p.slot_of[q];
      s_slot[threadIdx.x] = (s >= 0 && (int64_t)s < p.record_capacity) ? s : -1;
    }
    own_e = p.topk_idx[q];
    own_w = __float_as_uint(p.topk_weights[q]);
    if (SLOTS != kSlotsFused) {
      s_expert[threadIdx.x] = own_e;
      reinterpret_cast<int32_t*>(img + oi)[threadIdx.x] = own_e;
      reinterpret_cast<uint32_t*>(img + ow)[threadIdx.x] = own_w;
    }
  }
  zero_bytes(img, oi + 4 * k, ow);
  zero_bytes(img, ow + 4 * k, op);
  zero_bytes(img, op + p.payload_bytes, os);
  zero_bytes(img, os + p.scale_bytes, body);

  if (SLOTS == kSlotsFused) {
    const int hist_off = (body + (kQuant ? p.in_row_bytes : 0) + 15) & ~15;
    fused_layout(*lp, t, reinterpret_cast<int*>(img + hist_off), s_slot, p.record_capacity);
    if (threadIdx.x < k) {
      s_expert[threadIdx.x] = own_e;
      reinterpret_cast<int32_t*>(img + oi)[threadIdx.x] = own_e;
      reinterpret_cast<uint32_t*>(img + ow)[threadIdx.x] = own_w;
    }
  }

  cp_async_wait_all();
  __syncthreads();
  if (OUT_KIND == MOE_PAYLOAD_FP8_E4M3_B128) {
    quant_fp8(stage, p.hidden_size, img + op, reinterpret_cast<float*>(img + os));
  } else if (OUT_KIND == MOE_PAYLOAD_NVFP4_B16) {
    quant_nvfp4(stage, p.hidden_size, img + op, img + os);
  } else if (OUT_KIND == MOE_PAYLOAD_FP8_E4M3_UE8M0) {
    quant_fp8_ue8m0(stage, p.hidden_size, img + op, img + os);
  }

  fence_proxy_async_smem();
  if (SLOTS == kSlotsEarly) {
    pdl_wait();  // the layout has completed: slot_of is final
    pdl_trigger();
    if (threadIdx.x < k) {
      const int s = p.slot_of[(int64_t)t * k + threadIdx.x];
      s_slot[threadIdx.x] = (s >= 0 && (int64_t)s < p.record_capacity) ? s : -1;
    }
  }
  __syncthreads();

  if (threadIdx.x < k) {
    const int j = threadIdx.x;
    const int s = s_slot[j];
    if (s >= 0) {
      uint8_t* rec = p.records + (size_t)s * p.record_bytes;
      st_v4(rec, make_uint4((uint32_t)t, (uint32_t)j, (uint32_t)s_expert[j], 0u));
      bulk_store_s2g_evict_first(rec + 16, img, (uint32_t)body, l2_evict_first_policy());
      bulk_commit();
      bulk_wait_read_all();
    }
  }
}

// Eight resident blocks per SM need at most 32 registers a thread; the NVFP4
// quantiser would spill there, so it keeps six (40 registers).
template <int OUT_KIND, bool EARLY = false>
__global__ void __launch_bounds__(kDispatchThreads, OUT_KIND == MOE_PAYLOAD_NVFP4_B16 ? 6 : 8)
    k_dispatch(DispatchParams p) {
  dispatch_token<OUT_KIND, EARLY ? kSlotsEarly : kSlotsAfterWait>(p, nullptr);
}

// Layout and dispatch of a small routing in one launch (decode sizes: at most
// kFusedMaxPairs pairs, so at most that many blocks).
template <int OUT_KIND>
__global__ void __launch_bounds__(kDispatchThreads, 4) k_layout_dispatch_small(DispatchParams p, LayoutParams lp) {
  dispatch_token<OUT_KIND, kSlotsFused>(p, &lp);
}

// One record per (token, destination rank) instead of per (token, expert)
// (DeepEP Buffer::intranode_dispatch): the payload is built once in shared
// memory exactly as above; thread r then writes the record for rank r at
// send_head[t, r]. Its first segment (record bytes [0, off_payload)) is
//   header: int32 src_token, int32 rank, int32 number of local pairs, int32 0
//   ids:    topk_idx[t, j] - r*E/R for experts on rank r, else -1
//   weights: topk_weights[t, j] for experts on rank r, else 0
// (padding zero), written with 16-byte stores; payload and scales go to the
// bulk-copy engine.
template <int OUT_KIND>
__global__ void __launch_bounds__(kDispatchThreads)
    k_dispatch_ranks(DispatchParams p, const int32_t* send_head, int num_ranks, int experts_per_rank) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(128) uint8_t img[];  // record bytes [off_payload, record_bytes)
  __shared__ int s_ids[MOE_MAX_TOPK];
  __shared__ uint32_t s_w[MOE_MAX_TOPK];
  __shared__ int s_head[MOE_MAX_RANKS];
  const int t = blockIdx.x;
  const int k = p.topk;
  const int tail = p.record_bytes - p.off_payload;
  const int os = p.off_scales - p.off_payload;
  constexpr bool kQuant = OUT_KIND == MOE_PAYLOAD_FP8_E4M3_B128 || OUT_KIND == MOE_PAYLOAD_NVFP4_B16 ||
                          OUT_KIND == MOE_PAYLOAD_FP8_E4M3_UE8M0;
  uint8_t* stage = img + tail;
  const uint8_t* row = p.hidden + (size_t)t * p.in_row_bytes;
  if (kQuant) {
    copy_g2s_async(stage, row, p.in_row_bytes / 16);
  } else {
    copy_g2s_async(img, row, p.payload_bytes / 16);
    if (OUT_KIND == MOE_PAYLOAD_RAW && p.scale_bytes > 0)
      copy_g2s_async(img + os, p.scales + (size_t)t * p.in_scale_bytes, p.scale_bytes / 16);
  }
  if (threadIdx.x < k) {
    const int64_t q = (int64_t)t * k + threadIdx.x;
    s_ids[threadIdx.x] = p.topk_idx[q];
    s_w[threadIdx.x] = __float_as_uint(p.topk_weights[q]);
  }
  // the token's receive slots, loaded while the row is in flight
  if (threadIdx.x < num_ranks) s_head[threadIdx.x] = send_head[(int64_t)t * num_ranks + threadIdx.x];
  zero_bytes(img, p.payload_bytes, os);
  zero_bytes(img, os + p.scale_bytes, tail);
  cp_async_wait_all();
  __syncthreads();
  if (OUT_KIND == MOE_PAYLOAD_FP8_E4M3_B128) {
    quant_fp8(stage, p.hidden_size, img, reinterpret_cast<float*>(img + os));
  } else if (OUT_KIND == MOE_PAYLOAD_NVFP4_B16) {
    quant_nvfp4(stage, p.hidden_size, img, img + os);
  } else if (OUT_KIND == MOE_PAYLOAD_FP8_E4M3_UE8M0) {
    quant_fp8_ue8m0(stage, p.hidden_size, img, img + os);
  }
  fence_proxy_async_smem();
  __syncthreads();

  if (threadIdx.x < num_ranks) {
    const int r = threadIdx.x;
    const int s = s_head[r];
    if (s >= 0 && (int64_t)s < p.record_capacity) {
      const int lo = r * experts_per_rank, hi = lo + experts_per_rank;
      int nlocal = 0;
      for (int j = 0; j < k; ++j) nlocal += (s_ids[j] >= lo && s_ids[j] < hi) ? 1 : 0;
      const int pad_k = (p.off_weights - p.off_ids) / 4;
      uint8_t* rec = p.records + (size_t)s * p.record_bytes;
      for (int v = 0; v < p.off_payload / 16; ++v) {
        uint32_t wv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int w = v * 4 + i;
          uint32_t val = 0;
          if (w < 4) {
            val = w == 0 ? (uint32_t)t : w == 1 ? (uint32_t)r : w == 2 ? (uint32_t)nlocal : 0u;
          } else if (w < 4 + pad_k) {
            const int j = w - 4;
            if (j < k) {
              const int e = s_ids[j];
              val = (uint32_t)((e >= lo && e < hi) ? e - lo : -1);
            }
          } else {
            const int j = w - 4 - pad_k;
            if (j < k) val = (s_ids[j] >= lo && s_ids[j] < hi) ? s_w[j] : 0u;
          }
          wv[i] = val;
        }
        st_v4(rec + 16 * v, make_uint4(wv[0], wv[1], wv[2], wv[3]));
      }
      bulk_store_s2g_evict_first(rec + p.off_payload, img, (uint32_t)tail, l2_evict_first_policy());
      bulk_commit();
      bulk_wait_read_all();
    }
  }
}

// Payload and scales only, into two fixed-capacity, expert-major arrays (the
// low-latency receive buffers of DeepEP Buffer::low_latency_dispatch):
// pair (t, j) goes to row pos = slot_of[t, j] of x_out [rows, payload_bytes]
// and of scales_out [rows, scale_bytes rounded up to 16] (pad bytes zero). The payload is built once per token
// in shared memory as above; thread j issues the two bulk stores.
// EARLY (moe_layout_ll_dispatch only): as in k_dispatch_ranks, the payload is
// built before griddepcontrol.wait and the positions read after it.
template <int OUT_KIND, bool EARLY = false>
__global__ void __launch_bounds__(kDispatchThreads)
    k_dispatch_packed(DispatchParams p, uint8_t* x_out, uint8_t* scales_out, int64_t rows) {
  if (!EARLY) {
    pdl_wait();
    pdl_trigger();
  }
  extern __shared__ __align__(128) uint8_t img[];  // payload | scales | staged row
  __shared__ int s_pos[MOE_MAX_TOPK];
  const int t = blockIdx.x;
  const int k = p.topk;
  const int pb = p.payload_bytes, sb = p.scale_bytes;
  const int sbp = (sb + 15) & ~15;  // scale rows are padded to 16 bytes (zeros)
  constexpr bool kQuant = OUT_KIND == MOE_PAYLOAD_FP8_E4M3_B128 || OUT_KIND == MOE_PAYLOAD_NVFP4_B16 ||
                          OUT_KIND == MOE_PAYLOAD_FP8_E4M3_UE8M0;
  uint8_t* stage = img + pb + sbp;
  const uint8_t* row = p.hidden + (size_t)t * p.in_row_bytes;
  if (kQuant) {
    copy_g2s_async(stage, row, p.in_row_bytes / 16);
  } else {
    copy_g2s_async(img, row, pb / 16);
    if (OUT_KIND == MOE_PAYLOAD_RAW && sb > 0)
      copy_g2s_async(img + pb, p.scales + (size_t)t * p.in_scale_bytes, sb / 16);
  }
  if (!EARLY && threadIdx.x < k) {
    const int pos = p.slot_of[(int64_t)t * k + threadIdx.x];
    s_pos[threadIdx.x] = (pos >= 0 && (int64_t)pos < rows) ? pos : -1;
  }
  zero_bytes(img, pb + sb, pb + sbp);
  cp_async_wait_all();
  __syncthreads();
  if (OUT_KIND == MOE_PAYLOAD_FP8_E4M3_B128) {
    quant_fp8(stage, p.hidden_size, img, reinterpret_cast<float*>(img + pb));
  } else if (OUT_KIND == MOE_PAYLOAD_NVFP4_B16) {
    quant_nvfp4(stage, p.hidden_size, img, img + pb);
  } else if (OUT_KIND == MOE_PAYLOAD_FP8_E4M3_UE8M0) {
    quant_fp8_ue8m0(stage, p.hidden_size, img, img + pb);
  }
  fence_proxy_async_smem();
  if (EARLY) {
    pdl_wait();  // the layout has completed: the positions are final
    pdl_trigger();
    if (threadIdx.x < k) {
      const int pos = p.slot_of[(int64_t)t * k + threadIdx.x];
      s_pos[threadIdx.x] = (pos >= 0 && (int64_t)pos < rows) ? pos : -1;
    }
  }
  __syncthreads();
  if (threadIdx.x < k) {
    const int pos = s_pos[threadIdx.x];
    if (pos >= 0) {
      const uint64_t pol = l2_evict_first_policy();
      bulk_store_s2g_evict_first(x_out + (size_t)pos * pb, img, (uint32_t)pb, pol);
      if (sb > 0) bulk_store_s2g_evict_first(scales_out + (size_t)pos * sbp, img + pb, (uint32_t)sbp, pol);
      bulk_commit();
      bulk_wait_read_all();
    }
  }
}

}  // namespace

template <bool EARLY>
const void* dispatch_kernel(int out_kind) {
  switch (out_kind) {
    case MOE_PAYLOAD_BF16: return (const void*)k_dispatch<MOE_PAYLOAD_BF16, EARLY>;
    case MOE_PAYLOAD_FP8_E4M3_B128: return (const void*)k_dispatch<MOE_PAYLOAD_FP8_E4M3_B128, EARLY>;
    case MOE_PAYLOAD_NVFP4_B16: return (const void*)k_dispatch<MOE_PAYLOAD_NVFP4_B16, EARLY>;
    case MOE_PAYLOAD_FP8_E4M3_UE8M0: return (const void*)k_dispatch<MOE_PAYLOAD_FP8_E4M3_UE8M0, EARLY>;
    default: return (const void*)k_dispatch<MOE_PAYLOAD_RAW, EARLY>;
  }
}

cudaError_t launch_dispatch(const DispatchParams& p, int in_kind, int out_kind, cudaStream_t s,
                            bool after_layout) {
  (void)in_kind;
  const bool quant = out_kind == MOE_PAYLOAD_FP8_E4M3_B128 || out_kind == MOE_PAYLOAD_NVFP4_B16 ||
                     out_kind == MOE_PAYLOAD_FP8_E4M3_UE8M0;
  const size_t smem = (size_t)(p.record_bytes - 16) + (quant ? (size_t)p.in_row_bytes : 0);
  // the early form only when the stream's previous kernel is our layout and
  // the launch may overlap it
  const void* fn = after_layout && pdl_enabled() ? dispatch_kernel<true>(out_kind)
                                                 : dispatch_kernel<false>(out_kind);
  cudaError_t err = ensure_dynamic_smem(fn, smem);
  if (err != cudaSuccess) return err;
  DispatchParams q = p;
  void* args[] = {&q};
  return launch_pdl(fn, dim3((unsigned)p.num_tokens), dim3(kDispatchThreads), smem, s, args);
}

namespace {
size_t layout_dispatch_small_smem(const DispatchParams& p, int out_kind, int num_experts) {
  const bool quant = out_kind == MOE_PAYLOAD_FP8_E4M3_B128 || out_kind == MOE_PAYLOAD_NVFP4_B16 ||
                     out_kind == MOE_PAYLOAD_FP8_E4M3_UE8M0;
  const size_t hist_off = ((size_t)(p.record_bytes - 16) + (quant ? (size_t)p.in_row_bytes : 0) + 15) & ~(size_t)15;
  return hist_off + 4 * ((size_t)fused_hist_ints(num_experts) + (size_t)p.num_tokens * p.topk);
}
// the pair limit: kFusedDefaultPairs, or MOE_FUSED_LAYOUT=n (0 = never, at most kFusedMaxPairs)
int fused_pair_limit() {
  static const int limit = [] {
    const char* v = getenv("MOE_FUSED_LAYOUT");
    if (!v || !*v) return kFusedDefaultPairs;
    const long n = strtol(v, nullptr, 10);
    return (int)(n < 0 ? 0 : n > kFusedMaxPairs ? kFusedMaxPairs : n);
  }();
  return limit;
}
constexpr size_t kFusedMaxSmem = 200 * 1024;
}  // namespace

bool layout_dispatch_small_fits(const DispatchParams& p, int out_kind, int num_experts) {
  return p.num_tokens > 0 && (int64_t)p.num_tokens * p.topk <= fused_pair_limit() &&
         num_experts <= MOE_MAX_EXPERTS && layout_dispatch_small_smem(p, out_kind, num_experts) <= kFusedMaxSmem;
}

cudaError_t launch_layout_dispatch_small(const DispatchParams& p, const LayoutParams& lp, int out_kind,
                                         cudaStream_t s) {
  const size_t smem = layout_dispatch_small_smem(p, out_kind, lp.num_experts);
  const void* fn = nullptr;
  switch (out_kind) {
    case MOE_PAYLOAD_BF16: fn = (const void*)k_layout_dispatch_small<MOE_PAYLOAD_BF16>; break;
    case MOE_PAYLOAD_FP8_E4M3_B128: fn = (const void*)k_layout_dispatch_small<MOE_PAYLOAD_FP8_E4M3_B128>; break;
    case MOE_PAYLOAD_NVFP4_B16: fn = (const void*)k_layout_dispatch_small<MOE_PAYLOAD_NVFP4_B16>; break;
    case MOE_PAYLOAD_FP8_E4M3_UE8M0: fn = (const void*)k_layout_dispatch_small<MOE_PAYLOAD_FP8_E4M3_UE8M0>; break;
    default: fn = (const void*)k_layout_dispatch_small<MOE_PAYLOAD_RAW>; break;
  }
  cudaError_t err = ensure_dynamic_smem(fn, smem);
  if (err != cudaSuccess) return err;
  DispatchParams q = p;
  LayoutParams l = lp;
  void* args[] = {&q, &l};
  return launch_pdl(fn, dim3((unsigned)p.num_tokens), dim3(kDispatchThreads), smem, s, args);
}

template <bool EARLY>
const void* dispatch_packed_kernel(int out_kind) {
  switch (out_kind) {
    case MOE_PAYLOAD_BF16: return (const void*)k_dispatch_packed<MOE_PAYLOAD_BF16, EARLY>;
    case MOE_PAYLOAD_FP8_E4M3_B128: return (const void*)k_dispatch_packed<MOE_PAYLOAD_FP8_E4M3_B128, EARLY>;
    case MOE_PAYLOAD_NVFP4_B16: return (const void*)k_dispatch_packed<MOE_PAYLOAD_NVFP4_B16, EARLY>;
    case MOE_PAYLOAD_FP8_E4M3_UE8M0: return (const void*)k_dispatch_packed<MOE_PAYLOAD_FP8_E4M3_UE8M0, EARLY>;
    default: return (const void*)k_dispatch_packed<MOE_PAYLOAD_RAW, EARLY>;
  }
}

cudaError_t launch_dispatch_ranks(const DispatchParams& p, int out_kind, const int32_t* send_head,
                                  int num_ranks, int experts_per_rank, cudaStream_t s) {
  const bool quant = out_kind == MOE_PAYLOAD_FP8_E4M3_B128 || out_kind == MOE_PAYLOAD_NVFP4_B16 ||
                     out_kind == MOE_PAYLOAD_FP8_E4M3_UE8M0;
  const size_t smem = (size_t)(p.record_bytes - p.off_payload) + (quant ? (size_t)p.in_row_bytes : 0);
  const void* fn = nullptr;
  switch (out_kind) {
    case MOE_PAYLOAD_BF16: fn = (const void*)k_dispatch_ranks<MOE_PAYLOAD_BF16>; break;
    case MOE_PAYLOAD_FP8_E4M3_B128: fn = (const void*)k_dispatch_ranks<MOE_PAYLOAD_FP8_E4M3_B128>; break;
    case MOE_PAYLOAD_NVFP4_B16: fn = (const void*)k_dispatch_ranks<MOE_PAYLOAD_NVFP4_B16>; break;
    case MOE_PAYLOAD_FP8_E4M3_UE8M0: fn = (const void*)k_dispatch_ranks<MOE_PAYLOAD_FP8_E4M3_UE8M0>; break;
    default: fn = (const void*)k_dispatch_ranks<MOE_PAYLOAD_RAW>; break;
  }
  cudaError_t err = ensure_dynamic_smem(fn, smem);
  if (err != cudaSuccess) return err;
  DispatchParams q = p;
  const int32_t* sh = send_head;
  int nr = num_ranks, epr = experts_per_rank;
  void* args[] = {&q, &sh, &nr, &epr};
  return launch_pdl(fn, dim3((unsigned)p.num_tokens), dim3(kDispatchThreads), smem, s, args);
}

cudaError_t launch_dispatch_packed(const DispatchParams& p, int out_kind, uint8_t* x_out,
                                   uint8_t* scales_out, int64_t rows, cudaStream_t s, bool after_layout) {
  const bool quant = out_kind == MOE_PAYLOAD_FP8_E4M3_B128 || out_kind == MOE_PAYLOAD_NVFP4_B16 ||
                     out_kind == MOE_PAYLOAD_FP8_E4M3_UE8M0;
  const size_t smem = (size_t)p.payload_bytes + (size_t)((p.scale_bytes + 15) & ~15) +
                      (quant ? (size_t)p.in_row_bytes : 0);
  const void* fn = after_layout && pdl_enabled() ? dispatch_packed_kernel<true>(out_kind)
                                                 : dispatch_packed_kernel<false>(out_kind);
  cudaError_t err = ensure_dynamic_smem(fn, smem);
  if (err != cudaSuccess) return err;
  DispatchParams q = p;
  uint8_t* xo = x_out;
  uint8_t* so = scales_out;
  int64_t r = rows;
  void* args[] = {&q, &xo, &so, &r};
  return launch_pdl(fn, dim3((unsigned)p.num_tokens), dim3(kDispatchThreads), smem, s, args);
}

}  // namespace moe
