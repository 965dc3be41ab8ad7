// slots.cu -- the tensor-major rank-slot packing of the decode all-gather and
// the padded-token mask (vLLM compare view ds-exp-2...ds-exp-ag):
//  * moe_allgather.cu "Host launcher" (make_desc): each rank's slot holds its
//    2-4 tensors (top-k ids, weights, hidden payload, scales) one after the
//    other at 16-byte-aligned offsets; every tensor's byte size is a multiple
//    of 16. The gathered output of tensor i is all ranks' tensor i in rank
//    order.
//  * all2all.py mask_topk_ids: ids of tokens at or past num_actual_tokens (a
//    device scalar, so the call stays valid inside a replayed CUDA graph) are
//    set to -1.
// Pack and unpack are pure 16-byte vector copies: one launch covers every
// tensor of every rank, each thread moving whole 16-byte vectors with
// read-only streaming loads.
#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int kSlotThreads = 256;

struct SlotArgs {
  const uint8_t* src[MOE_MAX_SLOT_TENSORS];
  uint8_t* dst[MOE_MAX_SLOT_TENSORS];
  int64_t bytes[MOE_MAX_SLOT_TENSORS];   // per rank
  int64_t offset[MOE_MAX_SLOT_TENSORS];  // in a slot
  int64_t slot_bytes;
  int64_t vec_per_rank;                  // 16-byte vectors of one rank, all tensors
  int num_tensors, num_ranks;
};

// Vector v of rank r lies in tensor i at byte b = v*16 - offset[i] (tensors
// are contiguous in the slot since each size is a multiple of 16).
template <bool PACK>
__global__ void __launch_bounds__(kSlotThreads) k_slots(SlotArgs a) {
  pdl_wait();
  pdl_trigger();
  const int64_t total = a.vec_per_rank * a.num_ranks;
  for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < total;
       g += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = g / a.vec_per_rank;
    const int64_t byte = (g - r * a.vec_per_rank) * 16;
    int i = 0;
    while (i + 1 < a.num_tensors && byte >= a.offset[i + 1]) ++i;
    const int64_t in_t = byte - a.offset[i];
    const int64_t slot_pos = r * a.slot_bytes + byte;
    const int64_t t_pos = r * a.bytes[i] + in_t;
    if (PACK)
      st_v4(a.dst[0] + slot_pos, ld_stream_v4(a.src[i] + t_pos));
    else
      st_v4(a.dst[i] + t_pos, ld_stream_v4(a.src[0] + slot_pos));
  }
}

__global__ void k_mask_topk_ids(int32_t* ids, int64_t total, int topk, const int32_t* num_actual) {
  pdl_wait();
  pdl_trigger();
  const int na = *num_actual;  // a negative count masks every token
  const int64_t first = (int64_t)(na > 0 ? na : 0) * topk;
  for (int64_t i = first + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x)
    ids[i] = -1;
}

int blocks_for(int64_t work, int threads) {
  int dev = 0, sms = 148;
  if (!current_device(&dev, &sms)) sms = 148;
  int64_t b = (work + threads - 1) / threads;
  const int64_t cap = (int64_t)sms * 8;
  if (b > cap) b = cap;
  return b < 1 ? 1 : (int)b;
}

}  // namespace

cudaError_t launch_slots(bool pack, const void* const* src, void* const* dst,
                         const moe_slot_desc_t* d, const int64_t* offsets, int64_t slot_bytes,
                         cudaStream_t s) {
  SlotArgs a = {};
  a.num_tensors = d->num_tensors;
  a.num_ranks = d->num_ranks;
  a.slot_bytes = slot_bytes;
  a.vec_per_rank = slot_bytes / 16;
  for (int i = 0; i < d->num_tensors; ++i) {
    a.bytes[i] = d->bytes[i];
    a.offset[i] = offsets[i];
    a.src[i] = (const uint8_t*)src[pack ? i : 0];
    a.dst[i] = (uint8_t*)dst[pack ? 0 : i];
  }
  const int64_t work = a.vec_per_rank * a.num_ranks;
  if (work == 0) return cudaSuccess;
  const int blocks = blocks_for(work, kSlotThreads);
  void* args[] = {&a};
  return launch_pdl(pack ? (const void*)k_slots<true> : (const void*)k_slots<false>, dim3(blocks),
                    dim3(kSlotThreads), 0, s, args);
}

cudaError_t launch_mask_topk_ids(int32_t* ids, int64_t total, int topk, const int32_t* num_actual,
                                 cudaStream_t s) {
  if (total == 0) return cudaSuccess;
  int32_t* a0 = ids;
  int64_t a1 = total;
  int a2 = topk;
  const int32_t* a3 = num_actual;
  void* args[] = {&a0, &a1, &a2, &a3};
  return launch_pdl((const void*)k_mask_topk_ids, dim3(blocks_for(total, 256)), dim3(256), 0, s, args);
}

}  // namespace moe
