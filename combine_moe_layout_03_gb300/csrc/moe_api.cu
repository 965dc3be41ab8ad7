// moe_api.cu -- the extern "C" entry points of libmoe.so (declared and
// documented in include/moe.h): argument validation on the host, then the
// launches. Nothing here allocates device memory or synchronises, except
// moe_layout_status.
#include <stdlib.h>
#include <string.h>

#include <mutex>
#include <vector>

#include "moe_internal.cuh"

namespace moe {

bool pdl_enabled() {
  static const bool on = [] {
    const char* v = getenv("MOE_PDL");
    return !(v && v[0] == '0' && v[1] == '\0');
  }();
  return on;
}

namespace {
constexpr int kMaxDevices = 64;
std::once_flag g_sm_once[kMaxDevices];
int g_sm_count[kMaxDevices];
std::mutex g_smem_mutex;
struct SmemLimit {
  const void* fn;
  int dev;
  size_t bytes;
};
std::vector<SmemLimit> g_smem_limits;
}  // namespace

bool current_device(int* dev, int* sms) {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) {
    cudaGetLastError();
    return false;
  }
  std::call_once(g_sm_once[d], [d] {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d) != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    g_sm_count[d] = n;
  });
  if (g_sm_count[d] <= 0) return false;
  *dev = d;
  *sms = g_sm_count[d];
  return true;
}

cudaError_t ensure_dynamic_smem(const void* fn, size_t bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaGetLastError();
  std::lock_guard<std::mutex> lock(g_smem_mutex);
  for (SmemLimit& l : g_smem_limits) {
    if (l.fn == fn && l.dev == dev) {
      if (l.bytes >= bytes) return cudaSuccess;
      cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
      if (e == cudaSuccess) l.bytes = bytes;
      return e;
    }
  }
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) g_smem_limits.push_back({fn, dev, bytes});
  return e;
}

cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       void** args, unsigned cluster_x) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  if (pdl_enabled()) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster_x > 0) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace moe

namespace {

inline bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }
inline int pad16(int x) { return (x + 15) / 16 * 16; }

// Shape checks shared by every call. Returns MOE_OK or an error code.
int check_desc(const moe_desc_t* d) {
  if (!d) return MOE_ERR_INVALID_ARG;
  if (d->num_tokens < 0 || d->topk < 1 || d->num_experts < 1 || d->num_ranks < 1)
    return MOE_ERR_SHAPE;
  if (d->topk > MOE_MAX_TOPK || d->num_experts > MOE_MAX_EXPERTS || d->num_ranks > MOE_MAX_RANKS)
    return MOE_ERR_SHAPE;
  if (d->num_experts % d->num_ranks != 0) return MOE_ERR_SHAPE;
  if ((int64_t)d->num_tokens * d->topk >= ((int64_t)1 << 31)) return MOE_ERR_SHAPE;
  return MOE_OK;
}

int record_layout(const moe_desc_t* d, moe_record_layout_t* o) {
  int rc = check_desc(d);
  if (rc != MOE_OK) return rc;
  int pb = 0, sb = 0;
  const int H = d->hidden;
  if (d->in_kind == MOE_PAYLOAD_RAW && d->out_kind == MOE_PAYLOAD_RAW) {
    if (d->raw_payload_bytes < 0 || d->raw_scale_bytes < 0) return MOE_ERR_SHAPE;
    if (d->raw_payload_bytes > MOE_MAX_RAW_BYTES || d->raw_scale_bytes > MOE_MAX_RAW_BYTES)
      return MOE_ERR_SHAPE;
    if (d->raw_payload_bytes % 16 || d->raw_scale_bytes % 16) return MOE_ERR_ALIGNMENT;
    pb = d->raw_payload_bytes;
    sb = d->raw_scale_bytes;
  } else if (d->in_kind == MOE_PAYLOAD_BF16) {
    if (H < 1 || H > MOE_MAX_HIDDEN_DISPATCH) return MOE_ERR_SHAPE;
    switch (d->out_kind) {
      case MOE_PAYLOAD_BF16:
        if (H % 8) return MOE_ERR_SHAPE;
        pb = 2 * H;
        break;
      case MOE_PAYLOAD_FP8_E4M3_B128:
        if (H % 128) return MOE_ERR_SHAPE;
        pb = H;
        sb = H / 128 * 4;
        break;
      case MOE_PAYLOAD_NVFP4_B16:
        if (H % 16) return MOE_ERR_SHAPE;
        pb = H / 2;
        sb = H / 16;
        break;
      case MOE_PAYLOAD_FP8_E4M3_UE8M0:
        if (H % 128) return MOE_ERR_SHAPE;
        pb = H;
        sb = H / 128;
        break;
      default:
        return MOE_ERR_INVALID_ARG;
    }
  } else {
    return MOE_ERR_INVALID_ARG;
  }
  o->off_ids = 16;
  o->off_weights = o->off_ids + pad16(4 * d->topk);
  o->off_payload = o->off_weights + pad16(4 * d->topk);
  o->off_scales = o->off_payload + pad16(pb);
  o->record_bytes = o->off_scales + pad16(sb);
  o->payload_bytes = pb;
  o->scale_bytes = sb;
  return MOE_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// Validates moe_layout's arguments and fills its launch parameters (also
// for num_tokens == 0, when only the counts and the status word are written).
int layout_params(const moe_desc_t* desc, const int32_t* topk_idx, int32_t* tokens_per_expert,
                  int32_t* tokens_per_rank, uint8_t* is_token_in_rank, int32_t* expert_offset,
                  int32_t* rank_offset, int32_t* slot_of, int32_t* src_of_slot, void* workspace,
                  size_t ws_bytes, moe::LayoutParams* p) {
  int rc = check_desc(desc);
  if (rc != MOE_OK) return rc;
  const int N = desc->num_tokens, E = desc->num_experts, R = desc->num_ranks;
  if (!tokens_per_expert || !tokens_per_rank || !expert_offset || !rank_offset || !workspace)
    return MOE_ERR_INVALID_ARG;
  if (N > 0 && (!topk_idx || !is_token_in_rank || !slot_of)) return MOE_ERR_INVALID_ARG;
  const void* ints[] = {topk_idx, tokens_per_expert, tokens_per_rank, expert_offset,
                        rank_offset, slot_of, src_of_slot};
  for (const void* q : ints)
    if (!aligned(q, 4)) return MOE_ERR_ALIGNMENT;
  if (!aligned(workspace, 256)) return MOE_ERR_ALIGNMENT;
  const size_t need = moe::layout_workspace_bytes(N, E, R);
  if (ws_bytes < need) return MOE_ERR_CAPACITY;
  uint8_t* ws = (uint8_t*)workspace;
  p->topk_idx = topk_idx;
  p->tokens_per_expert = tokens_per_expert;
  p->tokens_per_rank = tokens_per_rank;
  p->is_token_in_rank = is_token_in_rank;
  p->expert_offset = expert_offset;
  p->rank_offset = rank_offset;
  p->slot_of = slot_of;
  p->src_of_slot = src_of_slot;
  p->num_tokens = N;
  p->topk = desc->topk;
  p->num_experts = E;
  p->num_ranks = R;
  p->experts_per_rank = E / R;
  p->tokens_per_chunk = moe::kLayoutTokensPerChunk;
  p->num_chunks = (N + moe::kLayoutTokensPerChunk - 1) / moe::kLayoutTokensPerChunk;
  p->status = (int32_t*)ws;
  p->chunk_hist = (int32_t*)(ws + 256);
  p->chunk_rank = p->chunk_hist + (size_t)p->num_chunks * E;
  p->chunk_flag = p->chunk_rank + (size_t)p->num_chunks * R;
  p->send_head = nullptr;  // no receive layout unless moe_layout_ranks asks for it
  p->recv_src_idx = nullptr;
  p->recv_offset = nullptr;
  p->recv_tokens_per_expert = nullptr;
  p->expert_alignment = 1;
  return MOE_OK;
}

}  // namespace

extern "C" {

const char* moe_strerror(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument (null pointer, kind or mode)";
    case MOE_ERR_ALIGNMENT: return "pointer or segment not 16-byte aligned";
    case MOE_ERR_SHAPE: return "shape outside the supported limits";
    case MOE_ERR_CAPACITY: return "a caller buffer is too small";
    case MOE_ERR_CUDA: return "a CUDA launch or copy failed";
    case MOE_ERR_DEVICE_IDS: return "an expert id was outside [-1, num_experts)";
    case MOE_ERR_TOO_LARGE: return "shape needs more scratch than moe_layout_noalloc's fixed array";
    case MOE_ERR_TIMEOUT: return "a bounded device wait gave up";
    default: return "unknown status";
  }
}

int moe_record_layout(const moe_desc_t* desc, moe_record_layout_t* out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  return record_layout(desc, out);
}

size_t moe_workspace_size(const moe_desc_t* desc) {
  if (check_desc(desc) != MOE_OK) return 0;
  return moe::layout_workspace_bytes(desc->num_tokens, desc->num_experts, desc->num_ranks);
}

int moe_layout(const moe_desc_t* desc, const int32_t* topk_idx, int32_t* tokens_per_expert,
               int32_t* tokens_per_rank, uint8_t* is_token_in_rank, int32_t* expert_offset,
               int32_t* rank_offset, int32_t* slot_of, int32_t* src_of_slot, void* workspace,
               size_t ws_bytes, moe_stream_t stream) {
  moe::LayoutParams p;
  int rc = layout_params(desc, topk_idx, tokens_per_expert, tokens_per_rank, is_token_in_rank,
                         expert_offset, rank_offset, slot_of, src_of_slot, workspace, ws_bytes, &p);
  if (rc != MOE_OK) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  if (p.num_tokens == 0) {  // nothing routed: zero counts and offsets
    const int E = p.num_experts, R = p.num_ranks;
    cudaError_t e = cudaMemsetAsync(tokens_per_expert, 0, (size_t)E * 4, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(tokens_per_rank, 0, (size_t)R * 4, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(expert_offset, 0, (size_t)(E + 1) * 4, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(rank_offset, 0, (size_t)(R + 1) * 4, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(p.status, 0, 4, s);  // status = MOE_OK
    return cuda_status(e);
  }
  return cuda_status(moe::launch_layout(p, s));
}

int moe_layout_ranks(const moe_desc_t* desc, const int32_t* topk_idx, int32_t* tokens_per_expert,
                     int32_t* tokens_per_rank, uint8_t* is_token_in_rank, int32_t* expert_offset,
                     int32_t* rank_offset, int32_t* slot_of, int32_t* src_of_slot, int32_t expert_alignment,
                     int32_t* send_head, int32_t* recv_src_idx, int32_t* recv_offset,
                     int32_t* recv_tokens_per_expert, void* workspace, size_t ws_bytes, moe_stream_t stream) {
  moe::LayoutParams p;
  int rc = layout_params(desc, topk_idx, tokens_per_expert, tokens_per_rank, is_token_in_rank,
                         expert_offset, rank_offset, slot_of, src_of_slot, workspace, ws_bytes, &p);
  if (rc != MOE_OK) return rc;
  const int N = p.num_tokens;
  if (expert_alignment < 1 || !recv_offset || !recv_tokens_per_expert) return MOE_ERR_INVALID_ARG;
  if (N > 0 && !send_head) return MOE_ERR_INVALID_ARG;
  const void* ints[] = {send_head, recv_src_idx, recv_offset, recv_tokens_per_expert};
  for (const void* q : ints)
    if (!aligned(q, 4)) return MOE_ERR_ALIGNMENT;
  cudaStream_t s = (cudaStream_t)stream;
  bool done = false;
  if (N > 0) {
    p.send_head = send_head;
    p.recv_src_idx = recv_src_idx;
    p.recv_offset = recv_offset;
    p.recv_tokens_per_expert = recv_tokens_per_expert;
    p.expert_alignment = expert_alignment;
    if (moe::launch_layout(p, s, &done) != cudaSuccess) return MOE_ERR_CUDA;
  } else {
    rc = moe_layout(desc, topk_idx, tokens_per_expert, tokens_per_rank, is_token_in_rank, expert_offset,
                    rank_offset, slot_of, src_of_slot, workspace, ws_bytes, stream);
    if (rc != MOE_OK) return rc;
  }
  if (done) return MOE_OK;
  // the layout ran as two kernels: the receive layout follows as its own kernel
  moe::RankLayoutParams rp;
  rp.is_token_in_rank = is_token_in_rank;
  rp.tokens_per_rank = tokens_per_rank;
  rp.tokens_per_expert = tokens_per_expert;
  rp.send_head = send_head;
  rp.recv_src_idx = recv_src_idx;
  rp.recv_offset = recv_offset;
  rp.recv_tokens_per_expert = recv_tokens_per_expert;
  rp.num_tokens = N;
  rp.num_ranks = p.num_ranks;
  rp.num_experts = p.num_experts;
  rp.expert_alignment = expert_alignment;
  return cuda_status(moe::launch_rank_layout(rp, s));
}

int moe_layout_ll(const moe_desc_t* desc, const int32_t* topk_idx, int32_t* tokens_per_expert,
                  int32_t* tokens_per_rank, uint8_t* is_token_in_rank, int32_t* expert_offset,
                  int32_t* rank_offset, int32_t* slot_of, int32_t* src_of_slot, int32_t max_tokens_per_rank,
                  int32_t* ll_slot_of, int32_t* src_info, int64_t* layout_range, int32_t* recv_count,
                  void* workspace, size_t ws_bytes, moe_stream_t stream) {
  moe::LayoutParams p;
  int rc = layout_params(desc, topk_idx, tokens_per_expert, tokens_per_rank, is_token_in_rank,
                         expert_offset, rank_offset, slot_of, src_of_slot, workspace, ws_bytes, &p);
  if (rc != MOE_OK) return rc;
  const int N = p.num_tokens, R = p.num_ranks;
  if (max_tokens_per_rank < 1 || N % R || N / R > max_tokens_per_rank) return MOE_ERR_SHAPE;
  const int64_t cap = (int64_t)R * max_tokens_per_rank;
  if ((int64_t)p.num_experts * cap >= ((int64_t)1 << 31)) return MOE_ERR_SHAPE;
  if (!src_info || !layout_range || !recv_count) return MOE_ERR_INVALID_ARG;
  if (N > 0 && (!ll_slot_of || !src_of_slot)) return MOE_ERR_INVALID_ARG;
  const void* ints[] = {ll_slot_of, src_info, recv_count};
  for (const void* q : ints)
    if (!aligned(q, 4)) return MOE_ERR_ALIGNMENT;
  if (!aligned(layout_range, 8)) return MOE_ERR_ALIGNMENT;
  cudaStream_t s = (cudaStream_t)stream;
  bool done = false;
  if (N > 0) {
    p.ll_slot_of = ll_slot_of;
    p.src_info = src_info;
    p.layout_range = layout_range;
    p.recv_count = recv_count;
    p.ll_capacity = cap;
    p.ll_tokens_per_rank = N / R;
    if (moe::launch_layout(p, s, &done) != cudaSuccess) return MOE_ERR_CUDA;
  } else {
    rc = moe_layout(desc, topk_idx, tokens_per_expert, tokens_per_rank, is_token_in_rank, expert_offset,
                    rank_offset, slot_of, src_of_slot, workspace, ws_bytes, stream);
    if (rc != MOE_OK) return rc;
  }
  if (done) return MOE_OK;
  // the cluster launch did not take it: the fixed-capacity layout as its own kernel
  return moe_ll_layout(desc, max_tokens_per_rank, topk_idx, slot_of, expert_offset, src_of_slot, ll_slot_of,
                       src_info, layout_range, recv_count, stream);
}

int moe_layout_status(const void* workspace, int32_t* status, moe_stream_t stream) {
  if (!workspace || !status) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  int32_t v = MOE_OK;
  cudaError_t e = cudaMemcpyAsync(&v, workspace, 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  *status = v;
  return MOE_OK;
}

int moe_device_status(int32_t* status, int clear) {
  if (!status) return MOE_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  return moe::read_device_status(status, clear != 0);
}

int moe_set_wait_limit_ns(uint64_t ns) {
  moe::set_wait_limit_ns(ns);
  return MOE_OK;
}

}  // extern "C"

namespace {

// Validates moe_dispatch's arguments and fills its launch parameters.
// Returns MOE_OK (p ready), or an error; *empty is set when there is no work.
int dispatch_params(const moe_desc_t* desc, const int32_t* topk_idx, const float* topk_weights,
                    const void* hidden, const void* scales, const int32_t* slot_of, void* records,
                    size_t records_bytes, moe::DispatchParams* p, bool* empty) {
  moe_record_layout_t lay;
  int rc = record_layout(desc, &lay);
  if (rc != MOE_OK) return rc;
  const int N = desc->num_tokens;
  *empty = N == 0;
  if (N == 0) return MOE_OK;
  const bool raw = desc->out_kind == MOE_PAYLOAD_RAW;
  if (!topk_idx || !topk_weights || !hidden || !slot_of || !records) return MOE_ERR_INVALID_ARG;
  if (raw && lay.scale_bytes > 0 && !scales) return MOE_ERR_INVALID_ARG;
  if (!aligned(topk_idx, 4) || !aligned(topk_weights, 4) || !aligned(slot_of, 4))
    return MOE_ERR_ALIGNMENT;
  if (!aligned(hidden, 16) || !aligned(records, 16) || (raw && scales && !aligned(scales, 16)))
    return MOE_ERR_ALIGNMENT;
  if (records_bytes < (size_t)lay.record_bytes) return MOE_ERR_CAPACITY;
  p->topk_idx = topk_idx;
  p->topk_weights = topk_weights;
  p->hidden = (const uint8_t*)hidden;
  p->scales = (const uint8_t*)scales;
  p->slot_of = slot_of;
  p->records = (uint8_t*)records;
  p->record_capacity = (int64_t)(records_bytes / (size_t)lay.record_bytes);
  p->num_tokens = N;
  p->topk = desc->topk;
  p->hidden_size = desc->hidden;
  p->in_row_bytes = raw ? desc->raw_payload_bytes : 2 * desc->hidden;
  p->in_scale_bytes = raw ? desc->raw_scale_bytes : 0;
  p->record_bytes = lay.record_bytes;
  p->off_ids = lay.off_ids;
  p->off_weights = lay.off_weights;
  p->off_payload = lay.off_payload;
  p->off_scales = lay.off_scales;
  p->payload_bytes = lay.payload_bytes;
  p->scale_bytes = lay.scale_bytes;
  return MOE_OK;
}

}  // namespace

extern "C" {

int moe_dispatch(const moe_desc_t* desc, const int32_t* topk_idx, const float* topk_weights,
                 const void* hidden, const void* scales, const int32_t* slot_of, void* records,
                 size_t records_bytes, moe_stream_t stream) {
  moe::DispatchParams p;
  bool empty = false;
  int rc = dispatch_params(desc, topk_idx, topk_weights, hidden, scales, slot_of, records,
                           records_bytes, &p, &empty);
  if (rc != MOE_OK || empty) return rc;
  return cuda_status(moe::launch_dispatch(p, desc->in_kind, desc->out_kind, (cudaStream_t)stream));
}

int moe_layout_dispatch(const moe_desc_t* desc, const int32_t* topk_idx, const float* topk_weights,
                        const void* hidden, const void* scales, int32_t* tokens_per_expert,
                        int32_t* tokens_per_rank, uint8_t* is_token_in_rank, int32_t* expert_offset,
                        int32_t* rank_offset, int32_t* slot_of, int32_t* src_of_slot,
                        void* workspace, size_t ws_bytes, void* records, size_t records_bytes,
                        moe_stream_t stream) {
  moe::DispatchParams p;
  bool empty = false;
  int rc = dispatch_params(desc, topk_idx, topk_weights, hidden, scales, slot_of, records,
                           records_bytes, &p, &empty);
  if (rc != MOE_OK) return rc;
  if (!empty && moe::layout_dispatch_small_fits(p, desc->out_kind, desc->num_experts)) {
    moe::LayoutParams lp;
    rc = layout_params(desc, topk_idx, tokens_per_expert, tokens_per_rank, is_token_in_rank,
                       expert_offset, rank_offset, slot_of, src_of_slot, workspace, ws_bytes, &lp);
    if (rc != MOE_OK) return rc;
    return cuda_status(moe::launch_layout_dispatch_small(p, lp, desc->out_kind, (cudaStream_t)stream));
  }
  rc = moe_layout(desc, topk_idx, tokens_per_expert, tokens_per_rank, is_token_in_rank,
                  expert_offset, rank_offset, slot_of, src_of_slot, workspace, ws_bytes, stream);
  if (rc != MOE_OK || empty) return rc;
  return cuda_status(
      moe::launch_dispatch(p, desc->in_kind, desc->out_kind, (cudaStream_t)stream, true));
}

int moe_combine(const moe_desc_t* desc, int mode, const void* expert_out, int64_t expert_out_rows,
                const int32_t* topk_idx, const float* topk_weights, const int32_t* slot_of,
                void* out, moe_stream_t stream) {
  int rc = check_desc(desc);
  if (rc != MOE_OK) return rc;
  const int N = desc->num_tokens, H = desc->hidden, R = desc->num_ranks;
  if (mode != MOE_COMBINE_TOPK && mode != MOE_COMBINE_RANKS && mode != MOE_COMBINE_TOPK_RANKS)
    return MOE_ERR_INVALID_ARG;
  if (H < 8 || H % 8) return MOE_ERR_SHAPE;
  if (mode != MOE_COMBINE_TOPK && N % R) return MOE_ERR_SHAPE;
  if ((int64_t)H / 8 > (int64_t)65535 * 128) return MOE_ERR_SHAPE;
  if (N == 0) return MOE_OK;
  if (!expert_out || !out) return MOE_ERR_INVALID_ARG;
  if (!aligned(expert_out, 16) || !aligned(out, 16)) return MOE_ERR_ALIGNMENT;
  if (expert_out_rows < 0) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  if (mode == MOE_COMBINE_RANKS) {
    if (expert_out_rows < (int64_t)R * N) return MOE_ERR_CAPACITY;
    return cuda_status(moe::launch_combine_ranks((const uint8_t*)expert_out, (uint8_t*)out,
                                                 (int64_t)N, H, R, s));
  }
  if (!topk_weights || !slot_of) return MOE_ERR_INVALID_ARG;
  if (mode == MOE_COMBINE_TOPK_RANKS && !topk_idx) return MOE_ERR_INVALID_ARG;
  if (!aligned(topk_weights, 4) || !aligned(slot_of, 4) || !aligned(topk_idx, 4))
    return MOE_ERR_ALIGNMENT;
  moe::CombineParams p;
  p.expert_out = (const uint8_t*)expert_out;
  p.expert_out_rows = expert_out_rows;
  p.topk_idx = topk_idx;
  p.topk_weights = topk_weights;
  p.slot_of = slot_of;
  p.out = (uint8_t*)out;
  p.num_tokens = N;
  p.topk = desc->topk;
  p.hidden_size = H;
  p.num_ranks = R;
  p.experts_per_rank = desc->num_experts / R;
  p.group_by_rank = mode == MOE_COMBINE_TOPK_RANKS;
  return cuda_status(moe::launch_combine_topk(p, s));
}

int moe_combine_norm(const moe_desc_t* desc, int mode, const void* expert_out,
                     int64_t expert_out_rows, const int32_t* topk_idx, const float* topk_weights,
                     const int32_t* slot_of, const void* residual_in, const void* gamma, float eps,
                     void* normed_out, void* residual_out, moe_stream_t stream) {
  int rc = check_desc(desc);
  if (rc != MOE_OK) return rc;
  const int N = desc->num_tokens, H = desc->hidden, R = desc->num_ranks;
  if (mode != MOE_COMBINE_TOPK && mode != MOE_COMBINE_RANKS && mode != MOE_COMBINE_TOPK_RANKS)
    return MOE_ERR_INVALID_ARG;
  if (H < 8 || H % 8 || H > moe::kMaxHiddenNorm) return MOE_ERR_SHAPE;
  if (mode != MOE_COMBINE_TOPK && N % R) return MOE_ERR_SHAPE;
  if (!(eps >= 0.0f) || eps > 3.0e38f) return MOE_ERR_INVALID_ARG;
  if (N == 0) return MOE_OK;
  if (!expert_out || !residual_in || !gamma || !normed_out || !residual_out) return MOE_ERR_INVALID_ARG;
  if (!aligned(expert_out, 16) || !aligned(residual_in, 16) || !aligned(gamma, 16) ||
      !aligned(normed_out, 16) || !aligned(residual_out, 16))
    return MOE_ERR_ALIGNMENT;
  if (expert_out_rows < 0) return MOE_ERR_INVALID_ARG;
  if (mode == MOE_COMBINE_RANKS) {
    if (expert_out_rows < (int64_t)R * N) return MOE_ERR_CAPACITY;
  } else {
    if (!topk_weights || !slot_of) return MOE_ERR_INVALID_ARG;
    if (mode == MOE_COMBINE_TOPK_RANKS && !topk_idx) return MOE_ERR_INVALID_ARG;
    if (!aligned(topk_weights, 4) || !aligned(slot_of, 4) || !aligned(topk_idx, 4))
      return MOE_ERR_ALIGNMENT;
  }
  moe::CombineNormParams p;
  p.c.expert_out = (const uint8_t*)expert_out;
  p.c.expert_out_rows = expert_out_rows;
  p.c.topk_idx = topk_idx;
  p.c.topk_weights = topk_weights;
  p.c.slot_of = slot_of;
  p.c.out = nullptr;
  p.c.num_tokens = N;
  p.c.topk = desc->topk;
  p.c.hidden_size = H;
  p.c.num_ranks = R;
  p.c.experts_per_rank = desc->num_experts / R;
  p.c.group_by_rank = mode == MOE_COMBINE_TOPK_RANKS;
  p.mode = mode;
  p.residual_in = (const uint8_t*)residual_in;
  p.gamma = (const uint8_t*)gamma;
  p.normed_out = (uint8_t*)normed_out;
  p.residual_out = (uint8_t*)residual_out;
  p.eps = eps;
  return cuda_status(moe::launch_combine_norm(p, (cudaStream_t)stream));
}

int moe_rank_layout(const moe_desc_t* desc, const uint8_t* is_token_in_rank,
                    const int32_t* tokens_per_rank, const int32_t* tokens_per_expert,
                    int32_t expert_alignment, int32_t* send_head, int32_t* recv_src_idx,
                    int32_t* recv_offset, int32_t* recv_tokens_per_expert, moe_stream_t stream) {
  int rc = check_desc(desc);
  if (rc != MOE_OK) return rc;
  if (expert_alignment < 1) return MOE_ERR_INVALID_ARG;
  const int N = desc->num_tokens, R = desc->num_ranks, E = desc->num_experts;
  if (!tokens_per_rank || !tokens_per_expert || !recv_offset || !recv_tokens_per_expert)
    return MOE_ERR_INVALID_ARG;
  if (N > 0 && (!is_token_in_rank || !send_head)) return MOE_ERR_INVALID_ARG;
  const void* ints[] = {tokens_per_rank, tokens_per_expert, send_head, recv_src_idx, recv_offset,
                        recv_tokens_per_expert};
  for (const void* q : ints)
    if (!aligned(q, 4)) return MOE_ERR_ALIGNMENT;
  moe::RankLayoutParams p;
  p.is_token_in_rank = is_token_in_rank;
  p.tokens_per_rank = tokens_per_rank;
  p.tokens_per_expert = tokens_per_expert;
  p.send_head = send_head;
  p.recv_src_idx = recv_src_idx;
  p.recv_offset = recv_offset;
  p.recv_tokens_per_expert = recv_tokens_per_expert;
  p.num_tokens = N;
  p.num_ranks = R;
  p.num_experts = E;
  p.expert_alignment = expert_alignment;
  return cuda_status(moe::launch_rank_layout(p, (cudaStream_t)stream));
}

}  // extern "C"

namespace {

// Validates moe_dispatch_ranks' arguments and fills its launch parameters;
// *empty is set when there is no work.
int dispatch_ranks_params(const moe_desc_t* desc, const int32_t* topk_idx, const float* topk_weights,
                          const void* hidden, const void* scales, const int32_t* send_head, void* records,
                          size_t records_bytes, moe::DispatchParams* p, bool* empty) {
  moe_record_layout_t lay;
  int rc = record_layout(desc, &lay);
  if (rc != MOE_OK) return rc;
  const int N = desc->num_tokens;
  *empty = N == 0;
  if (N == 0) return MOE_OK;
  const bool raw = desc->out_kind == MOE_PAYLOAD_RAW;
  if (!topk_idx || !topk_weights || !hidden || !send_head || !records) return MOE_ERR_INVALID_ARG;
  if (raw && lay.scale_bytes > 0 && !scales) return MOE_ERR_INVALID_ARG;
  if (!aligned(topk_idx, 4) || !aligned(topk_weights, 4) || !aligned(send_head, 4))
    return MOE_ERR_ALIGNMENT;
  if (!aligned(hidden, 16) || !aligned(records, 16) || (raw && scales && !aligned(scales, 16)))
    return MOE_ERR_ALIGNMENT;
  if (records_bytes < (size_t)lay.record_bytes) return MOE_ERR_CAPACITY;
  p->topk_idx = topk_idx;
  p->topk_weights = topk_weights;
  p->hidden = (const uint8_t*)hidden;
  p->scales = (const uint8_t*)scales;
  p->slot_of = nullptr;
  p->records = (uint8_t*)records;
  p->record_capacity = (int64_t)(records_bytes / (size_t)lay.record_bytes);
  p->num_tokens = N;
  p->topk = desc->topk;
  p->hidden_size = desc->hidden;
  p->in_row_bytes = raw ? desc->raw_payload_bytes : 2 * desc->hidden;
  p->in_scale_bytes = raw ? desc->raw_scale_bytes : 0;
  p->record_bytes = lay.record_bytes;
  p->off_ids = lay.off_ids;
  p->off_weights = lay.off_weights;
  p->off_payload = lay.off_payload;
  p->off_scales = lay.off_scales;
  p->payload_bytes = lay.payload_bytes;
  p->scale_bytes = lay.scale_bytes;
  return MOE_OK;
}

}  // namespace

extern "C" {

int moe_dispatch_ranks(const moe_desc_t* desc, const int32_t* topk_idx,
                       const float* topk_weights, const void* hidden, const void* scales,
                       const int32_t* send_head, void* records, size_t records_bytes,
                       moe_stream_t stream) {
  moe::DispatchParams p;
  bool empty = false;
  int rc = dispatch_ranks_params(desc, topk_idx, topk_weights, hidden, scales, send_head, records,
                                 records_bytes, &p, &empty);
  if (rc != MOE_OK || empty) return rc;
  return cuda_status(moe::launch_dispatch_ranks(p, desc->out_kind, send_head, desc->num_ranks,
                                                desc->num_experts / desc->num_ranks,
                                                (cudaStream_t)stream));
}

int moe_combine_gather_ranks(const moe_desc_t* desc, const void* recv_out, int64_t recv_rows,
                             const int32_t* send_head, void* out, moe_stream_t stream) {
  int rc = check_desc(desc);
  if (rc != MOE_OK) return rc;
  const int N = desc->num_tokens, H = desc->hidden;
  if (H < 8 || H % 8) return MOE_ERR_SHAPE;
  if (N == 0) return MOE_OK;
  if (!recv_out || !send_head || !out || recv_rows < 0) return MOE_ERR_INVALID_ARG;
  if (!aligned(recv_out, 16) || !aligned(out, 16) || !aligned(send_head, 4))
    return MOE_ERR_ALIGNMENT;
  moe::RankCombineParams p;
  p.recv_out = (const uint8_t*)recv_out;
  p.rows = recv_rows;
  p.send_head = send_head;
  p.out = (uint8_t*)out;
  p.num_tokens = N;
  p.num_ranks = desc->num_ranks;
  p.hidden_size = H;
  return cuda_status(moe::launch_combine_gather_ranks(p, (cudaStream_t)stream));
}

int moe_ll_layout(const moe_desc_t* desc, int32_t max_tokens_per_rank, const int32_t* topk_idx,
                  const int32_t* slot_of, const int32_t* expert_offset,
                  const int32_t* src_of_slot, int32_t* ll_slot_of, int32_t* src_info,
                  int64_t* layout_range, int32_t* recv_count, moe_stream_t stream) {
  int rc = check_desc(desc);
  if (rc != MOE_OK) return rc;
  const int N = desc->num_tokens, R = desc->num_ranks;
  if (max_tokens_per_rank < 1 || N % R || N / R > max_tokens_per_rank) return MOE_ERR_SHAPE;
  const int64_t cap = (int64_t)R * max_tokens_per_rank;
  if ((int64_t)desc->num_experts * cap >= ((int64_t)1 << 31)) return MOE_ERR_SHAPE;
  if (!expert_offset || !src_info || !layout_range || !recv_count) return MOE_ERR_INVALID_ARG;
  if (N > 0 && (!topk_idx || !slot_of || !src_of_slot || !ll_slot_of)) return MOE_ERR_INVALID_ARG;
  const void* ints[] = {topk_idx, slot_of, expert_offset, src_of_slot, ll_slot_of, src_info,
                        recv_count};
  for (const void* q : ints)
    if (!aligned(q, 4)) return MOE_ERR_ALIGNMENT;
  if (!aligned(layout_range, 8)) return MOE_ERR_ALIGNMENT;
  moe::LlLayoutParams p;
  p.topk_idx = topk_idx;
  p.slot_of = slot_of;
  p.expert_offset = expert_offset;
  p.src_of_slot = src_of_slot;
  p.ll_slot_of = ll_slot_of;
  p.src_info = src_info;
  p.layout_range = layout_range;
  p.recv_count = recv_count;
  p.capacity = cap;
  p.num_tokens = N;
  p.topk = desc->topk;
  p.num_experts = desc->num_experts;
  p.num_ranks = R;
  return cuda_status(moe::launch_ll_layout(p, (cudaStream_t)stream));
}

}  // extern "C"

namespace {

// Validates moe_dispatch_ll's arguments and fills its launch parameters and
// the rows the output buffers hold; *empty is set when there is no work.
int dispatch_ll_params(const moe_desc_t* desc, const void* hidden, const void* scales,
                       const int32_t* ll_slot_of, void* x_out, size_t x_out_bytes, void* scales_out,
                       size_t scales_out_bytes, moe::DispatchParams* p, int64_t* rows_out, bool* empty) {
  moe_record_layout_t lay;
  int rc = record_layout(desc, &lay);
  if (rc != MOE_OK) return rc;
  if (lay.payload_bytes % 16) return MOE_ERR_SHAPE;
  const int64_t scale_row = (lay.scale_bytes + 15) / 16 * 16;  // padded scale rows
  const int N = desc->num_tokens;
  *empty = N == 0;
  if (N == 0) return MOE_OK;
  const bool raw = desc->out_kind == MOE_PAYLOAD_RAW;
  if (!hidden || !ll_slot_of || !x_out) return MOE_ERR_INVALID_ARG;
  if (lay.scale_bytes > 0 && !scales_out) return MOE_ERR_INVALID_ARG;
  if (raw && lay.scale_bytes > 0 && !scales) return MOE_ERR_INVALID_ARG;
  if (!aligned(ll_slot_of, 4) || !aligned(hidden, 16) || !aligned(x_out, 16) ||
      !aligned(scales_out, 16) || (raw && scales && !aligned(scales, 16)))
    return MOE_ERR_ALIGNMENT;
  if (lay.payload_bytes == 0) return MOE_ERR_SHAPE;
  int64_t rows = (int64_t)(x_out_bytes / (size_t)lay.payload_bytes);
  if (lay.scale_bytes > 0) {
    const int64_t srows = (int64_t)(scales_out_bytes / (size_t)scale_row);
    if (srows < rows) rows = srows;
  }
  *p = moe::DispatchParams{};
  p->hidden = (const uint8_t*)hidden;
  p->scales = (const uint8_t*)scales;
  p->slot_of = ll_slot_of;
  p->num_tokens = N;
  p->topk = desc->topk;
  p->hidden_size = desc->hidden;
  p->in_row_bytes = raw ? desc->raw_payload_bytes : 2 * desc->hidden;
  p->in_scale_bytes = raw ? desc->raw_scale_bytes : 0;
  p->payload_bytes = lay.payload_bytes;
  p->scale_bytes = lay.scale_bytes;
  *rows_out = rows;
  return MOE_OK;
}

}  // namespace

extern "C" {

int moe_dispatch_ll(const moe_desc_t* desc, const void* hidden, const void* scales,
                    const int32_t* ll_slot_of, void* x_out, size_t x_out_bytes, void* scales_out,
                    size_t scales_out_bytes, moe_stream_t stream) {
  moe::DispatchParams p;
  int64_t rows = 0;
  bool empty = false;
  int rc = dispatch_ll_params(desc, hidden, scales, ll_slot_of, x_out, x_out_bytes, scales_out,
                              scales_out_bytes, &p, &rows, &empty);
  if (rc != MOE_OK || empty) return rc;
  return cuda_status(moe::launch_dispatch_packed(p, desc->out_kind, (uint8_t*)x_out,
                                                 (uint8_t*)scales_out, rows, (cudaStream_t)stream));
}

int moe_layout_ll_dispatch(const moe_desc_t* desc, const int32_t* topk_idx, const void* hidden,
                           const void* scales, int32_t* tokens_per_expert, int32_t* tokens_per_rank,
                           uint8_t* is_token_in_rank, int32_t* expert_offset, int32_t* rank_offset,
                           int32_t* slot_of, int32_t* src_of_slot, int32_t max_tokens_per_rank,
                           int32_t* ll_slot_of, int32_t* src_info, int64_t* layout_range, int32_t* recv_count,
                           void* workspace, size_t ws_bytes, void* x_out, size_t x_out_bytes, void* scales_out,
                           size_t scales_out_bytes, moe_stream_t stream) {
  moe::DispatchParams p;
  int64_t rows = 0;
  bool empty = false;
  int rc = dispatch_ll_params(desc, hidden, scales, ll_slot_of, x_out, x_out_bytes, scales_out,
                              scales_out_bytes, &p, &rows, &empty);
  if (rc != MOE_OK) return rc;
  rc = moe_layout_ll(desc, topk_idx, tokens_per_expert, tokens_per_rank, is_token_in_rank, expert_offset,
                     rank_offset, slot_of, src_of_slot, max_tokens_per_rank, ll_slot_of, src_info, layout_range,
                     recv_count, workspace, ws_bytes, stream);
  if (rc != MOE_OK || empty) return rc;
  // the previous kernel is this call's own (layout or fixed-capacity layout)
  return cuda_status(moe::launch_dispatch_packed(p, desc->out_kind, (uint8_t*)x_out, (uint8_t*)scales_out,
                                                 rows, (cudaStream_t)stream, true));
}

int moe_combine_backward(const moe_desc_t* desc, const void* grad_out, const float* topk_weights,
                         const int32_t* slot_of, const void* expert_out, int64_t rows,
                         void* grad_expert_out, float* grad_weights, moe_stream_t stream) {
  int rc = check_desc(desc);
  if (rc != MOE_OK) return rc;
  const int N = desc->num_tokens, H = desc->hidden;
  if (H < 8 || H % 8) return MOE_ERR_SHAPE;
  if (rows < 0) return MOE_ERR_INVALID_ARG;
  if (N == 0) return MOE_OK;
  if (!grad_out || !topk_weights || !slot_of || !grad_expert_out) return MOE_ERR_INVALID_ARG;
  if (expert_out && !grad_weights) return MOE_ERR_INVALID_ARG;
  if (expert_out && expert_out == grad_expert_out) return MOE_ERR_INVALID_ARG;
  if (!aligned(grad_out, 16) || !aligned(grad_expert_out, 16) || !aligned(expert_out, 16) ||
      !aligned(topk_weights, 4) || !aligned(slot_of, 4) || !aligned(grad_weights, 4))
    return MOE_ERR_ALIGNMENT;
  moe::CombineBwdParams p;
  p.grad_out = (const uint8_t*)grad_out;
  p.topk_weights = topk_weights;
  p.slot_of = slot_of;
  p.expert_out = (const uint8_t*)expert_out;
  p.rows = rows;
  p.grad_expert_out = (uint8_t*)grad_expert_out;
  p.grad_weights = expert_out ? grad_weights : nullptr;
  p.num_tokens = N;
  p.topk = desc->topk;
  p.hidden_size = H;
  return cuda_status(moe::launch_combine_backward(p, (cudaStream_t)stream));
}

int moe_dispatch_backward(const moe_desc_t* desc, const void* grad_in, int64_t rows,
                          const int32_t* slot_of, void* grad_hidden, moe_stream_t stream) {
  int rc = check_desc(desc);
  if (rc != MOE_OK) return rc;
  const int N = desc->num_tokens, H = desc->hidden;
  if (H < 8 || H % 8) return MOE_ERR_SHAPE;
  if ((int64_t)H / 8 > (int64_t)65535 * 128) return MOE_ERR_SHAPE;
  if (rows < 0) return MOE_ERR_INVALID_ARG;
  if (N == 0) return MOE_OK;
  if (!grad_in || !slot_of || !grad_hidden) return MOE_ERR_INVALID_ARG;
  if (!aligned(grad_in, 16) || !aligned(grad_hidden, 16) || !aligned(slot_of, 4))
    return MOE_ERR_ALIGNMENT;
  moe::CombineParams p;
  p.expert_out = (const uint8_t*)grad_in;
  p.expert_out_rows = rows;
  p.topk_idx = nullptr;
  p.topk_weights = nullptr;  // unit weights
  p.slot_of = slot_of;
  p.out = (uint8_t*)grad_hidden;
  p.num_tokens = N;
  p.topk = desc->topk;
  p.hidden_size = H;
  p.num_ranks = desc->num_ranks;
  p.experts_per_rank = desc->num_experts / desc->num_ranks;
  p.group_by_rank = 0;
  return cuda_status(moe::launch_combine_topk(p, (cudaStream_t)stream));
}

int moe_combine_gather_ranks_backward(const moe_desc_t* desc, const void* grad_out,
                                      const int32_t* send_head, void* grad_recv,
                                      int64_t recv_rows, moe_stream_t stream) {
  int rc = check_desc(desc);
  if (rc != MOE_OK) return rc;
  const int N = desc->num_tokens, H = desc->hidden;
  if (H < 8 || H % 8) return MOE_ERR_SHAPE;
  if (recv_rows < 0) return MOE_ERR_INVALID_ARG;
  if (N == 0) return MOE_OK;
  if (!grad_out || !send_head || !grad_recv) return MOE_ERR_INVALID_ARG;
  if (!aligned(grad_out, 16) || !aligned(grad_recv, 16) || !aligned(send_head, 4))
    return MOE_ERR_ALIGNMENT;
  moe::RankCombineBwdParams p;
  p.grad_out = (const uint8_t*)grad_out;
  p.send_head = send_head;
  p.grad_recv = (uint8_t*)grad_recv;
  p.rows = recv_rows;
  p.num_tokens = N;
  p.num_ranks = desc->num_ranks;
  p.hidden_size = H;
  return cuda_status(moe::launch_gather_ranks_backward(p, (cudaStream_t)stream));
}

int moe_slot_layout(const moe_slot_desc_t* desc, int64_t* offsets, int64_t* slot_bytes) {
  if (!desc || !offsets || !slot_bytes) return MOE_ERR_INVALID_ARG;
  if (desc->num_tensors < 2 || desc->num_tensors > MOE_MAX_SLOT_TENSORS || desc->num_ranks < 1)
    return MOE_ERR_INVALID_ARG;
  int64_t cursor = 0;
  for (int i = 0; i < desc->num_tensors; ++i) {
    if (desc->bytes[i] < 0) return MOE_ERR_INVALID_ARG;
    if (desc->bytes[i] % 16) return MOE_ERR_ALIGNMENT;
    cursor = (cursor + 15) / 16 * 16;
    offsets[i] = cursor;
    cursor += desc->bytes[i];
  }
  *slot_bytes = cursor;
  return MOE_OK;
}

static int slots_call(bool pack, const moe_slot_desc_t* desc, const void* const* tensors_in,
                      void* const* tensors_out, const void* slots_in, void* slots_out,
                      moe_stream_t stream) {
  int64_t off[MOE_MAX_SLOT_TENSORS];
  int64_t sb = 0;
  int rc = moe_slot_layout(desc, off, &sb);
  if (rc != MOE_OK) return rc;
  const void* src[MOE_MAX_SLOT_TENSORS] = {};
  void* dst[MOE_MAX_SLOT_TENSORS] = {};
  if (pack) {
    if (!tensors_in || !slots_out) return MOE_ERR_INVALID_ARG;
    for (int i = 0; i < desc->num_tensors; ++i) {
      if (!tensors_in[i] && desc->bytes[i]) return MOE_ERR_INVALID_ARG;
      if (!aligned(tensors_in[i], 16)) return MOE_ERR_ALIGNMENT;
      src[i] = tensors_in[i];
    }
    if (!aligned(slots_out, 16)) return MOE_ERR_ALIGNMENT;
    dst[0] = slots_out;
  } else {
    if (!tensors_out || !slots_in) return MOE_ERR_INVALID_ARG;
    for (int i = 0; i < desc->num_tensors; ++i) {
      if (!tensors_out[i] && desc->bytes[i]) return MOE_ERR_INVALID_ARG;
      if (!aligned(tensors_out[i], 16)) return MOE_ERR_ALIGNMENT;
      dst[i] = tensors_out[i];
    }
    if (!aligned(slots_in, 16)) return MOE_ERR_ALIGNMENT;
    src[0] = slots_in;
  }
  return cuda_status(moe::launch_slots(pack, src, dst, desc, off, sb, (cudaStream_t)stream));
}

int moe_pack_slots(const moe_slot_desc_t* desc, const void* const* tensors, void* slots,
                   moe_stream_t stream) {
  return slots_call(true, desc, tensors, nullptr, nullptr, slots, stream);
}

int moe_unpack_slots(const moe_slot_desc_t* desc, const void* slots, void* const* tensors,
                     moe_stream_t stream) {
  return slots_call(false, desc, nullptr, tensors, slots, nullptr, stream);
}

int moe_mask_topk_ids(int32_t* topk_idx, int32_t num_tokens, int32_t topk,
                      const int32_t* num_actual_tokens, moe_stream_t stream) {
  if (num_tokens < 0 || topk < 1 || topk > MOE_MAX_TOPK) return MOE_ERR_SHAPE;
  if ((int64_t)num_tokens * topk >= ((int64_t)1 << 31)) return MOE_ERR_SHAPE;
  if (!num_actual_tokens || (num_tokens > 0 && !topk_idx)) return MOE_ERR_INVALID_ARG;
  if (!aligned(topk_idx, 4) || !aligned(num_actual_tokens, 4)) return MOE_ERR_ALIGNMENT;
  return cuda_status(moe::launch_mask_topk_ids(topk_idx, (int64_t)num_tokens * topk, topk,
                                               num_actual_tokens, (cudaStream_t)stream));
}

int moe_pack_record(const moe_desc_t* desc, int32_t src_token, int32_t slot_j, int32_t expert,
                    const int32_t* ids_row, const float* w_row, const void* payload_row,
                    const void* scales_row, void* record) {
  moe_record_layout_t lay;
  int rc = record_layout(desc, &lay);
  if (rc != MOE_OK) return rc;
  if (!ids_row || !w_row || !payload_row || !record) return MOE_ERR_INVALID_ARG;
  if (lay.scale_bytes > 0 && !scales_row) return MOE_ERR_INVALID_ARG;
  uint8_t* r = (uint8_t*)record;
  memset(r, 0, (size_t)lay.record_bytes);
  const int32_t hdr[4] = {src_token, slot_j, expert, 0};
  memcpy(r, hdr, 16);
  memcpy(r + lay.off_ids, ids_row, (size_t)desc->topk * 4);
  memcpy(r + lay.off_weights, w_row, (size_t)desc->topk * 4);
  memcpy(r + lay.off_payload, payload_row, (size_t)lay.payload_bytes);
  if (lay.scale_bytes > 0) memcpy(r + lay.off_scales, scales_row, (size_t)lay.scale_bytes);
  return MOE_OK;
}

int moe_unpack_record(const moe_desc_t* desc, const void* record, int32_t* src_token,
                      int32_t* slot_j, int32_t* expert, int32_t* ids_row, float* w_row,
                      void* payload_row, void* scales_row) {
  moe_record_layout_t lay;
  int rc = record_layout(desc, &lay);
  if (rc != MOE_OK) return rc;
  if (!record) return MOE_ERR_INVALID_ARG;
  const uint8_t* r = (const uint8_t*)record;
  int32_t hdr[4];
  memcpy(hdr, r, 16);
  if (src_token) *src_token = hdr[0];
  if (slot_j) *slot_j = hdr[1];
  if (expert) *expert = hdr[2];
  if (ids_row) memcpy(ids_row, r + lay.off_ids, (size_t)desc->topk * 4);
  if (w_row) memcpy(w_row, r + lay.off_weights, (size_t)desc->topk * 4);
  if (payload_row) memcpy(payload_row, r + lay.off_payload, (size_t)lay.payload_bytes);
  if (scales_row && lay.scale_bytes > 0) memcpy(scales_row, r + lay.off_scales, (size_t)lay.scale_bytes);
  return MOE_OK;
}

}  // extern "C"
