/*
 * moe.h -- C ABI of libmoe.so: MoE token dispatch and combine on one GPU.
 *
 * The library computes the data-parallel hot path of Mixture-of-Experts token
 * routing with expert-parallel ranks emulated as R regions of one GPU's
 * memory:
 *
 *   moe_layout    routing layout: per-expert and per-rank counts, prefix
 *                 offsets, the token-in-rank mask and a stable slot map
 *                 (DeepEP repository, csrc/deep_ep.cpp,
 *                 Buffer::get_dispatch_layout);
 *   moe_dispatch  one 16-byte-aligned record per (token, top-k) pair, grouped
 *                 by destination rank and expert, with the payload optionally
 *                 quantised to FP8 e4m3 per 128 channels or NVFP4 per 16
 *                 (DeepEP csrc/config.hpp LowLatencyLayout message: int4
 *                 header + payload + scales; Buffer::low_latency_dispatch
 *                 FP8 cast; vLLM compare view ds-exp-2...ds-exp-ag,
 *                 moe_allgather.cu "Host launcher": tensors packed at
 *                 16-byte-aligned offsets);
 *   moe_combine   the top-k weighted BF16 reduction back to token order and
 *                 the cross-rank sum a reduce-scatter performs (DeepEP
 *                 Buffer::low_latency_combine; ds-exp-ag moe_reduce_scatter.cu
 *                 "Lamport reduce-scatter kernel" phase 3; vLLM PR
 *                 "Eliminate staging from NCCL symmetric reduce-scatter",
 *                 Implementation).
 *
 * Further groups below: the fused combine + residual + RMSNorm; the
 * per-(token, rank) layout, dispatch and gathered combine of DeepEP's normal
 * kernels; the fixed-capacity, expert-major buffers of its low-latency
 * kernels; the backward of combine and dispatch; the decode all-gather's
 * rank-slot packing and padded-token mask; an allocation-free layout.
 *
 * Conventions
 *  - Every function returns an int status: MOE_OK (0) or a negative MOE_ERR_*
 *    code; moe_strerror() names it. Nothing throws, aborts or traps. Argument
 *    errors are found on the host before anything is launched.
 *  - All buffers belong to the caller. Device pointers are allocated and freed
 *    by the caller; the library allocates nothing, keeps no state between
 *    calls and never synchronises the stream (except moe_layout_status, which
 *    says so). Work is enqueued on the caller's stream.
 *  - moe_stream_t is a cudaStream_t passed as void*; NULL is the legacy
 *    default stream.
 *  - Kernels are launched with programmatic dependent launch: each one waits
 *    (griddepcontrol.wait) for the previous kernel in the stream to complete
 *    and its memory to be visible before it touches global memory, so it may
 *    become resident early and hide the launch gap, whatever ran before it.
 *    The environment variable MOE_PDL=0, read once per process, launches in
 *    plain stream order instead.
 *  - Integers in records are little-endian.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes -------------------------------------------------------- */
#define MOE_OK 0
#define MOE_ERR_INVALID_ARG (-1) /* NULL pointer, bad kind or mode, size < needed */
#define MOE_ERR_ALIGNMENT (-2)   /* pointer or segment not 16-byte aligned */
#define MOE_ERR_SHAPE (-3)       /* shape outside the supported limits below */
#define MOE_ERR_CAPACITY (-4)    /* a caller buffer is too small */
#define MOE_ERR_CUDA (-5)        /* a CUDA launch or copy failed */
#define MOE_ERR_DEVICE_IDS (-6)  /* (from moe_layout_status) an id was outside [-1, E) */
#define MOE_ERR_TOO_LARGE (-7)   /* moe_layout_noalloc: the shape needs more scratch than it has */
#define MOE_ERR_TIMEOUT (-8)     /* (from moe_device_status) a bounded device wait gave up */

typedef void* moe_stream_t;

/* ---- payload kinds ------------------------------------------------------- */
/* What the caller's hidden rows are (in_kind) and what records carry
 * (out_kind). Valid pairs: (BF16, BF16), (BF16, FP8_E4M3_B128),
 * (BF16, NVFP4_B16), (BF16, FP8_E4M3_UE8M0), (RAW, RAW). */
#define MOE_PAYLOAD_BF16 0          /* bf16 [H] per token, H*2 bytes */
#define MOE_PAYLOAD_FP8_E4M3_B128 1 /* e4m3 [H] + fp32 scale per 128 channels */
#define MOE_PAYLOAD_NVFP4_B16 2     /* e2m1 [H/2 bytes] + e4m3 scale byte per 16 */
#define MOE_PAYLOAD_RAW 3           /* opaque bytes copied as they are */
/* e4m3 [H] + one UE8M0 byte per 128 channels (DeepEP low_latency_dispatch
 * use_ue8m0 / round_scale: one byte per 128-channel group, four groups to an
 * int32, H/128 bytes in group order). Reading (no formula on the pages): the
 * scale is the least power of two 2^e >= max(amax, 1e-4)/448 (the quotient
 * in IEEE fp32), q = e4m3_rn(x * 2^-e) (exact scaling, never saturating),
 * byte = e + 127 (value 2^(byte-127)). */
#define MOE_PAYLOAD_FP8_E4M3_UE8M0 4

/* ---- combine modes -------------------------------------------------------- */
#define MOE_COMBINE_TOPK 0       /* top-k weighted reduction to token order */
#define MOE_COMBINE_RANKS 1      /* cross-rank sum of R BF16 partials */
#define MOE_COMBINE_TOPK_RANKS 2 /* top-k reduction grouped by rank, then summed */

/* ---- limits ----------------------------------------------------------------- */
#define MOE_MAX_TOPK 32
#define MOE_MAX_EXPERTS 1024
#define MOE_MAX_RANKS 64
#define MOE_MAX_HIDDEN_DISPATCH 16384 /* BF16/FP8/NVFP4 dispatch */
#define MOE_MAX_RAW_BYTES 65536       /* RAW payload and scale bytes each */

/* Shape and format of one call. num_tokens N >= 0; topk k in [1, 32];
 * num_experts E in [1, 1024]; num_ranks R in [1, 64] with E % R == 0; expert e
 * lives on rank e / (E/R) (DeepEP Buffer::low_latency_dispatch: E % R == 0,
 * E/R local experts per rank). N * k < 2^31.
 * hidden H: channels per token. BF16 rows need H % 8 == 0 (16-byte rows);
 * FP8 needs H % 128 == 0; NVFP4 needs H % 32 == 0 (16-byte packed rows).
 * For RAW, raw_payload_bytes and raw_scale_bytes are the bytes per token of
 * the caller's two tensors; each must be a multiple of 16 (ds-exp-ag
 * moe_allgather.cu make_desc rejects other sizes) and <= MOE_MAX_RAW_BYTES;
 * raw_scale_bytes may be 0 (no scales). H is then only informational. */
typedef struct {
  int32_t num_tokens;
  int32_t topk;
  int32_t num_experts;
  int32_t num_ranks;
  int32_t hidden;
  int32_t in_kind;
  int32_t out_kind;
  int32_t raw_payload_bytes;
  int32_t raw_scale_bytes;
} moe_desc_t;

/* Byte layout of one record. Every offset and record_bytes is a multiple of
 * 16; padding bytes are zero.
 *   [0, 16)                 header: int32 src_token, int32 j, int32 expert, int32 0
 *   [off_ids, +4k)          the token's whole top-k id row (int32)
 *   [off_weights, +4k)      the token's fp32 weight row
 *   [off_payload, +payload_bytes)  BF16 row | e4m3 bytes | packed e2m1 | raw | e4m3 bytes
 *   [off_scales, +scale_bytes)     none | fp32 per 128 | e4m3 byte per 16 | raw |
 *                                  UE8M0 byte per 128
 * NVFP4 packing: byte i holds element 2i in bits 0-3 and element 2i+1 in bits
 * 4-7; e2m1 code = sign << 3 | magnitude index into {0,.5,1,1.5,2,3,4,6}. */
typedef struct {
  int32_t record_bytes;
  int32_t off_ids;
  int32_t off_weights;
  int32_t off_payload;
  int32_t off_scales;
  int32_t payload_bytes;
  int32_t scale_bytes;
} moe_record_layout_t;

/* Text for a status code (static storage, never NULL). */
const char* moe_strerror(int status);

/* Host only. Fills *out for the record format of desc. Errors:
 * INVALID_ARG (NULL, bad kind pair), SHAPE (limits above). */
int moe_record_layout(const moe_desc_t* desc, moe_record_layout_t* out);

/* Host only. Bytes of device scratch that moe_layout needs for desc (0 if desc
 * is invalid). The workspace must be 256-byte aligned. Its contents need no
 * initialisation and are meaningful only to the library; the status word of
 * the last moe_layout call lives in it. */
size_t moe_workspace_size(const moe_desc_t* desc);

/* Routing layout (DeepEP Buffer::get_dispatch_layout outputs plus the slot
 * map of the pairs; -1 ids mean "no expert", as vLLM's mask_topk_ids writes
 * for padded tokens on the ds-exp-ag page).
 * Inputs (device): topk_idx int32 [N, k], row-major.
 * Outputs (device, caller-allocated, fully written):
 *   tokens_per_expert int32 [E]   pairs routed to each expert
 *   tokens_per_rank   int32 [R]   tokens with at least one pair on the rank
 *   is_token_in_rank  uint8 [N,R] 1/0
 *   expert_offset     int32 [E+1] exclusive prefix sum of tokens_per_expert;
 *                                 expert_offset[E] = P, the number of records
 *   rank_offset       int32 [R+1] expert_offset[r * E/R]; rank r's records are
 *                                 slots [rank_offset[r], rank_offset[r+1])
 *   slot_of           int32 [N,k] record slot of pair (t, j), -1 for id -1.
 *                                 Inside an expert's region slots follow
 *                                 ascending (t, j): a stable counting sort.
 *   src_of_slot       int32 [N*k] t*k+j of the pair in slot s, -1 for s >= P.
 *                                 May be NULL.
 * workspace: device, >= moe_workspace_size(desc) bytes, 256-byte aligned.
 * An id outside [-1, E) is treated as -1 and recorded in the workspace's
 * status word; read it with moe_layout_status. All int pointers must be
 * 4-byte aligned. Errors: INVALID_ARG, SHAPE, ALIGNMENT, CAPACITY (ws_bytes),
 * CUDA. */
int moe_layout(const moe_desc_t* desc, const int32_t* topk_idx, int32_t* tokens_per_expert,
               int32_t* tokens_per_rank, uint8_t* is_token_in_rank, int32_t* expert_offset,
               int32_t* rank_offset, int32_t* slot_of, int32_t* src_of_slot, void* workspace,
               size_t ws_bytes, moe_stream_t stream);

/* Copies the status word of the last moe_layout that used this workspace to
 * *status (MOE_OK or MOE_ERR_DEVICE_IDS) after synchronising the stream.
 * This is the only call that waits for the device. Errors: INVALID_ARG, CUDA. */
int moe_layout_status(const void* workspace, int32_t* status, moe_stream_t stream);

/* Status of the kernels that wait on shared-memory barriers (the pipelined
 * combine: expert rows brought into shared memory by bulk copies). Every
 * such wait is bounded: after 1 s it gives up, the kernel records
 * MOE_ERR_TIMEOUT in a device word of the library and returns, leaving the
 * context usable. No legitimate run reaches that limit, since the copies are
 * reads of the GPU's own memory. *status receives MOE_OK or MOE_ERR_TIMEOUT
 * for all launches on the current device since the last call with clear != 0
 * (which resets the word). It synchronises the device; it is not for a hot
 * loop. Errors: INVALID_ARG, CUDA. */
int moe_device_status(int32_t* status, int clear);

/* Test hook for the bounded waits above. Sets, for launches made after the
 * call, how long each such wait may last before it gives up: ns of wall time
 * (%globaltimer), clamped to the default of one second; ns = 0 restores the
 * default. With a budget far below a copy's latency (e.g. 1 ns) the waits
 * give up at once: the kernel records MOE_ERR_TIMEOUT for moe_device_status,
 * leaves the output rows it did not finish unwritten and returns, with the
 * context still usable. A block always waits, with the full second, for the
 * copies it issued before it exits, so no copy lands after it. Process-wide
 * (every device), host only, does not synchronise. Always returns MOE_OK. */
int moe_set_wait_limit_ns(uint64_t ns);

/* Permute and pack (dispatch). For every pair (t, j) with slot_of[t, j] >= 0
 * writes one record (moe_record_layout) to
 * records + slot_of[t, j] * record_bytes. The payload of a token is computed
 * once and copied into each of its records.
 * Inputs (device): topk_idx int32 [N,k]; topk_weights fp32 [N,k];
 *   hidden: bf16 [N,H] (in_kind BF16) or uint8 [N, raw_payload_bytes] (RAW);
 *   scales: uint8 [N, raw_scale_bytes] for RAW with raw_scale_bytes > 0, else
 *   ignored (may be NULL); slot_of int32 [N,k] from moe_layout.
 * Output (device): records, at least P * record_bytes bytes
 *   (records_bytes says how many the caller has; N*k*record_bytes is always
 *   enough). Slots not named by slot_of are not touched.
 * FP8 per 128 channels (the pages give no formula; reading): amax = max|x|,
 *   a = max(amax, 1e-4), scale = a/448, q = e4m3_rn_satfinite(x * (448/a)),
 *   both divisions IEEE fp32; stored scale is fp32.
 * NVFP4 per 16 (reading, no global scale): sc = e4m3_rn_satfinite(amax/6),
 *   d = value(sc), q = d == 0 ? 0 : e2m1_rn_satfinite(x / d).
 * hidden, scales and records must be 16-byte aligned. Errors: INVALID_ARG,
 * SHAPE, ALIGNMENT, CAPACITY, CUDA. */
int moe_dispatch(const moe_desc_t* desc, const int32_t* topk_idx, const float* topk_weights,
                 const void* hidden, const void* scales, const int32_t* slot_of, void* records,
                 size_t records_bytes, moe_stream_t stream);

/* moe_layout followed by moe_dispatch in one call: the same outputs, bit for
 * bit, as the two calls in sequence. Because the kernel before the dispatch
 * is then known to be this call's own layout kernel, which writes none of
 * the dispatch's inputs, the dispatch loads and quantises its token rows
 * while the layout still runs and reads only slot_of after it (programmatic
 * dependent launch; with MOE_PDL=0 the two run in plain order). A routing of
 * at most 2048 pairs (N*k; decode batches up to 256 tokens of top-8) runs as
 * a single kernel instead, each of whose blocks computes the layout from all
 * ids while its token row loads (MOE_FUSED_LAYOUT=0 in the environment keeps
 * the two kernels; MOE_FUSED_LAYOUT=p lowers the limit to p pairs). Arguments are those of the two calls; all of them are
 * checked before anything is launched. Errors: as moe_layout and
 * moe_dispatch. */
int moe_layout_dispatch(const moe_desc_t* desc, const int32_t* topk_idx, const float* topk_weights,
                        const void* hidden, const void* scales, int32_t* tokens_per_expert,
                        int32_t* tokens_per_rank, uint8_t* is_token_in_rank, int32_t* expert_offset,
                        int32_t* rank_offset, int32_t* slot_of, int32_t* src_of_slot,
                        void* workspace, size_t ws_bytes, void* records, size_t records_bytes,
                        moe_stream_t stream);

/* Combine.
 * MOE_COMBINE_TOPK: expert_out bf16 [P, H] holds the expert outputs in slot
 *   order; out bf16 [N, H] with
 *     out[t] = bf16_rn( fp32 fma chain over j ascending, slot_of[t,j] >= 0,
 *                       of topk_weights[t,j] * expert_out[slot_of[t,j]] )
 *   (fp32 accumulation and round-to-nearest-even BF16 output as in the
 *   ds-exp-ag reduce-scatter; ascending j is the reading taken).
 *   topk_idx may be NULL.
 * MOE_COMBINE_RANKS: expert_out bf16 [R][N][H] holds R partials; out bf16
 *   [N, H] = bf16_rn(sum over r ascending of float(partial_r)), fp32
 *   accumulation; rank q's reduce-scatter output is rows [qN/R, (q+1)N/R).
 *   Needs N % R == 0. topk_idx, topk_weights, slot_of may be NULL.
 * MOE_COMBINE_TOPK_RANKS: as TOPK, but for each rank r (ascending) the fp32
 *   partial over the pairs whose expert lives on rank r (fma chain, ascending
 *   j) is formed first and the partials are summed in fp32, ascending r, with
 *   one BF16 rounding at the end. Needs N % R == 0 and topk_idx.
 * expert_out and out must be 16-byte aligned; H % 8 == 0. expert_out_rows is
 *   the number of rows the caller's expert_out holds (P for the TOPK modes,
 *   R*N for RANKS); a slot outside it is a caller error that the kernels
 *   skip. Errors: INVALID_ARG, SHAPE, ALIGNMENT, CAPACITY, CUDA. */
int moe_combine(const moe_desc_t* desc, int mode, const void* expert_out, int64_t expert_out_rows,
                const int32_t* topk_idx, const float* topk_weights, const int32_t* slot_of,
                void* out, moe_stream_t stream);

/* Allocation-free routing layout. The pages have no counterpart to this entry
 * point: it is the same computation as moe_layout for callers that cannot
 * give the library device memory for scratch -- for example a plugin inside a
 * host program that owns every device allocation through its own pool, or a
 * service that fixes its device footprint at start-up and must not call
 * cudaMalloc afterwards.
 * Instead of a workspace it uses a fixed array of MOE_NOALLOC_SCRATCH_BYTES
 * (2 MiB) inside the library's device image. That array exists on every GPU
 * that loads the library and is held until the process exits. The call
 * allocates nothing.
 * Arguments and outputs are those of moe_layout, without workspace and
 * ws_bytes. status (device int32, may be NULL) receives MOE_OK or
 * MOE_ERR_DEVICE_IDS for this call, written on the stream.
 * Limit: the layout needs 256 + ceil(N/128) * (E + R + 1) * 4 bytes of
 * scratch (moe_workspace_size); larger shapes return MOE_ERR_TOO_LARGE. For
 * E = 256, R = 8 that allows N up to about 253,000 tokens.
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture. The address is kept for the life of the process:
 * resetting a device (cudaDeviceReset) while the library is loaded is not
 * supported, since the next call would use the old context's address.
 * Every call shares the one array and overwrites
 * what it reads, so nothing needs clearing, but calls that overlap on the GPU
 * (different streams, or unordered host threads) race on it.
 * Errors: INVALID_ARG, SHAPE, ALIGNMENT, TOO_LARGE, CUDA. */
#define MOE_NOALLOC_SCRATCH_BYTES (2u << 20)
int moe_layout_noalloc(const moe_desc_t* desc, const int32_t* topk_idx,
                       int32_t* tokens_per_expert, int32_t* tokens_per_rank,
                       uint8_t* is_token_in_rank, int32_t* expert_offset, int32_t* rank_offset,
                       int32_t* slot_of, int32_t* src_of_slot, int32_t* status,
                       moe_stream_t stream);

/* Combine fused with the residual add and RMSNorm that follow it in the layer
 * (vLLM compare view ds-exp-2...ds-exp-ag, moe_rs_fused.cu: reduce-scatter,
 * residual add and RMSNorm in one kernel; test_rs_fused.py rms_norm_ref).
 * mode and expert_out, expert_out_rows, topk_idx, topk_weights, slot_of are as
 * in moe_combine. For every token t and channel h:
 *   x[t,h]            = s[t,h] + float(residual_in[t,h])   (fp32)
 *   residual_out[t,h] = bf16_rn(x[t,h])
 *   normed_out[t,h]   = bf16_rn((x[t,h] * rsqrt(sum_h x[t,h]^2 / H + eps)) * gamma[h])
 * where s is the mode's combine in fp32 before its final rounding (the value
 * moe_combine would round). residual_out is exact; the normed output carries
 * the rounding of an fp32 sum of squares and of rsqrt (fp32, products in the
 * order written).
 * residual_in, normed_out, residual_out: bf16 [N, H]; gamma: bf16 [H]; all
 * device, 16-byte aligned. eps >= 0. H % 8 == 0 and H <= 16384.
 * Errors: INVALID_ARG, SHAPE, ALIGNMENT, CAPACITY, CUDA. */
int moe_combine_norm(const moe_desc_t* desc, int mode, const void* expert_out,
                     int64_t expert_out_rows, const int32_t* topk_idx, const float* topk_weights,
                     const int32_t* slot_of, const void* residual_in, const void* gamma, float eps,
                     void* normed_out, void* residual_out, moe_stream_t stream);

/* ---- one record per (token, destination rank) ----------------------------
 * The shape of DeepEP's normal (intranode) dispatch and combine (DeepEP
 * repository, csrc/deep_ep.cpp Buffer::intranode_dispatch /
 * Buffer::intranode_combine): a token is sent once to every rank r with
 * is_token_in_rank[t, r], not once per expert; each rank's experts then
 * produce one (locally reduced) row per received token, and combine sums the
 * ranks' rows back to token order. */

/* Receive layout per rank, from moe_layout's outputs. For rank r the received
 * tokens are the t with is_token_in_rank[t, r], in ascending t (virtual
 * source ranks own contiguous token ranges, so this is source-rank order):
 *   recv_offset [R+1]   exclusive prefix sum of tokens_per_rank
 *   send_head   [N,R]   receive slot of token t on rank r, recv_offset[r] + its
 *                       position among rank r's tokens; -1 if not sent
 *   recv_src_idx [N*R]  source token of each receive slot, -1 past the last
 *                       (may be NULL)
 *   recv_tokens_per_expert [E]  tokens_per_expert[e] rounded up to a multiple
 *                       of expert_alignment (>= 1), as DeepEP aligns its
 *                       per-expert receive counts for grouped GEMMs
 * Inputs: is_token_in_rank uint8 [N,R], tokens_per_rank int32 [R],
 * tokens_per_expert int32 [E] (device). Errors: INVALID_ARG, SHAPE,
 * ALIGNMENT, CUDA. */
int moe_rank_layout(const moe_desc_t* desc, const uint8_t* is_token_in_rank,
                    const int32_t* tokens_per_rank, const int32_t* tokens_per_expert,
                    int32_t expert_alignment, int32_t* send_head, int32_t* recv_src_idx,
                    int32_t* recv_offset, int32_t* recv_tokens_per_expert, moe_stream_t stream);

/* moe_layout and moe_rank_layout in one call (DeepEP repository,
 * csrc/deep_ep.cpp Buffer::get_dispatch_layout, then the receive layout of
 * Buffer::intranode_dispatch). Arguments are those of moe_layout, then
 * expert_alignment and the receive-layout outputs of moe_rank_layout (which
 * it computes from this call's layout); every output is the one the two
 * calls give. Where the layout runs as one cluster launch (every workload of
 * the pages), the receive layout is computed in that launch from the rank
 * masks and the per-block rank counts the cluster already exchanges; larger
 * shapes take the two kernels. Errors: those of the two calls. */
int moe_layout_ranks(const moe_desc_t* desc, const int32_t* topk_idx, int32_t* tokens_per_expert,
                     int32_t* tokens_per_rank, uint8_t* is_token_in_rank, int32_t* expert_offset,
                     int32_t* rank_offset, int32_t* slot_of, int32_t* src_of_slot, int32_t expert_alignment,
                     int32_t* send_head, int32_t* recv_src_idx, int32_t* recv_offset,
                     int32_t* recv_tokens_per_expert, void* workspace, size_t ws_bytes, moe_stream_t stream);


/* Dispatch with one record per (token, rank) at records + send_head[t, r] *
 * record_bytes (moe_record_layout's format and sizes). The payload and
 * scales are those of moe_dispatch. The first segment differs (reading: the
 * pages show DeepEP's interface, not its kernel):
 *   header  int32 src_token, int32 rank, int32 number of the token's pairs on
 *           the rank, int32 0
 *   ids     topk_idx[t, j] - r*E/R (the local expert id) for experts on rank
 *           r, else -1
 *   weights topk_weights[t, j] for experts on rank r, else 0
 * Errors: as moe_dispatch. */
int moe_dispatch_ranks(const moe_desc_t* desc, const int32_t* topk_idx,
                       const float* topk_weights, const void* hidden, const void* scales,
                       const int32_t* send_head, void* records, size_t records_bytes,
                       moe_stream_t stream);

/* Combine of per-rank rows: recv_out bf16 [recv_rows, H] holds one row per
 * receive slot (each rank's locally reduced expert output for the token);
 *   out[t] = bf16( sum over r ascending with send_head[t, r] >= 0 of
 *                  float(recv_out[send_head[t, r]]) )    (fp32, from +0)
 * out bf16 [N, H]. H % 8 == 0; recv_out and out 16-byte aligned. Slots at or
 * past recv_rows are skipped. Errors: INVALID_ARG, SHAPE, ALIGNMENT, CUDA. */
int moe_combine_gather_ranks(const moe_desc_t* desc, const void* recv_out, int64_t recv_rows,
                             const int32_t* send_head, void* out, moe_stream_t stream);

/* ---- fixed-capacity, expert-major receive buffers -------------------------
 * The low-latency layout of DeepEP (csrc/deep_ep.cpp
 * Buffer::low_latency_dispatch / low_latency_combine): every expert has room
 * for capacity = R * max_tokens_per_rank received tokens (packed_recv_x
 * [E_l, R * max_tokens, H] per rank; [E, capacity, ...] for all R ranks of one
 * GPU), so buffer sizes never depend on the routing and the calls need no
 * host-side counts. Source rank s owns tokens [s*T, (s+1)*T), T = N / R.
 * Reading (the pages show the interface, not the kernels): expert e's pairs
 * are packed compactly from position 0 in source-rank, then token, order --
 * the stable slot order of moe_layout within e. */

/* From moe_layout's outputs:
 *   ll_slot_of   int32 [N,k]       e * capacity + position of pair (t, j), or -1
 *                                  (id -1, or beyond the expert's capacity)
 *   src_info     int32 [E,capacity] token index within its source rank, -1 in
 *                                  unused positions
 *   layout_range int64 [E,R]       begin << 32 | count of expert e's pairs from
 *                                  source rank s
 *   recv_count   int32 [E]         pairs received by each expert (capped at
 *                                  capacity)
 * Needs N % R == 0 and N / R <= max_tokens_per_rank. The combine back is
 * moe_combine (TOPK) with slot_of = ll_slot_of and expert_out the
 * [E * capacity, H] expert outputs. Errors: INVALID_ARG, SHAPE, ALIGNMENT, CUDA. */
int moe_ll_layout(const moe_desc_t* desc, int32_t max_tokens_per_rank, const int32_t* topk_idx,
                  const int32_t* slot_of, const int32_t* expert_offset,
                  const int32_t* src_of_slot, int32_t* ll_slot_of, int32_t* src_info,
                  int64_t* layout_range, int32_t* recv_count, moe_stream_t stream);

/* moe_layout and moe_ll_layout in one call. Arguments are those of moe_layout
 * (src_of_slot required), then max_tokens_per_rank and the outputs of
 * moe_ll_layout, which it computes from this call's layout; every output is
 * the one the two calls give. Where the layout runs as one cluster launch and
 * a source rank's T = N / R tokens can be a whole number of its blocks (the
 * low-latency decode workload of the pages: 8 x 128 tokens), the fixed-capacity
 * layout is computed in that launch from the expert counts every block of the
 * cluster already holds; otherwise the two calls' kernels run in turn. Needs
 * N % R == 0 and N / R <= max_tokens_per_rank. Errors: those of the two calls. */
int moe_layout_ll(const moe_desc_t* desc, const int32_t* topk_idx, int32_t* tokens_per_expert,
                  int32_t* tokens_per_rank, uint8_t* is_token_in_rank, int32_t* expert_offset,
                  int32_t* rank_offset, int32_t* slot_of, int32_t* src_of_slot, int32_t max_tokens_per_rank,
                  int32_t* ll_slot_of, int32_t* src_info, int64_t* layout_range, int32_t* recv_count,
                  void* workspace, size_t ws_bytes, moe_stream_t stream);

/* moe_layout_ll then moe_dispatch_ll in one call: arguments are those of
 * moe_layout_ll followed by x_out, x_out_bytes, scales_out and
 * scales_out_bytes of moe_dispatch_ll (hidden and scales as there). The
 * dispatch's blocks load and quantise their rows while the layout kernels
 * still run (they write none of the rows) and read ll_slot_of once they have
 * completed. Every dispatch argument is checked before anything is launched.
 * Outputs and errors: those of the two calls. */
int moe_layout_ll_dispatch(const moe_desc_t* desc, const int32_t* topk_idx, const void* hidden,
                           const void* scales, int32_t* tokens_per_expert, int32_t* tokens_per_rank,
                           uint8_t* is_token_in_rank, int32_t* expert_offset, int32_t* rank_offset,
                           int32_t* slot_of, int32_t* src_of_slot, int32_t max_tokens_per_rank,
                           int32_t* ll_slot_of, int32_t* src_info, int64_t* layout_range, int32_t* recv_count,
                           void* workspace, size_t ws_bytes, void* x_out, size_t x_out_bytes, void* scales_out,
                           size_t scales_out_bytes, moe_stream_t stream);

/* Dispatch into the fixed-capacity buffers: the payload of moe_dispatch
 * (quantised once per token) goes to row ll_slot_of[t, j] of x_out
 * [E * capacity, payload_bytes] and its scales to the same row of scales_out
 * [E * capacity, scale_row] with scale_row = scale_bytes rounded up to a
 * multiple of 16, the pad bytes zero (row-major; scales_out may be NULL when
 * there are none). payload_bytes must be a multiple of 16. FP8 with fp32
 * scales has no pad when H % 512 == 0, as DeepEP's low-latency FP8 cast
 * requires; UE8M0 scales (H/128 bytes, 56 at H = 7168) are padded to 64.
 * x_out_bytes and scales_out_bytes give the buffers' sizes. Errors: as
 * moe_dispatch. */
int moe_dispatch_ll(const moe_desc_t* desc, const void* hidden, const void* scales,
                    const int32_t* ll_slot_of, void* x_out, size_t x_out_bytes, void* scales_out,
                    size_t scales_out_bytes, moe_stream_t stream);

/* ---- backward (training) ------------------------------------------------
 * DeepEP README, "Example use in model training or inference prefilling":
 * the backward of combine is a dispatch of the gradient through the cached
 * handle (the layout is not recomputed), and the backward of dispatch is a
 * combine. Here the "handle" is the slot map (slot_of, ll_slot_of or
 * send_head) the forward calls used. */

/* Backward of the top-k weighted combine out[t] = sum_j w[t,j] * y[slot_of[t,j]]
 * (moe_combine TOPK or TOPK_RANKS, which differ only in rounding order):
 *   grad_expert_out[slot_of[t,j]] = bf16_rn(w[t,j] * grad_out[t])  (fp32 product)
 *   grad_weights[t,j] = sum_h grad_out[t,h] * expert_out[slot_of[t,j], h]
 *                       (fp32 accumulation, fixed order; 0 for a pair with no slot)
 * grad_out bf16 [N, H]; expert_out bf16 [rows, H] or NULL (then no weight
 * gradient and grad_weights is ignored); grad_expert_out bf16 [rows, H], of
 * which only the rows some pair names are written; grad_weights fp32 [N, k].
 * Slots outside [0, rows) are skipped. The buffers must not overlap.
 * H % 8 == 0, bf16 buffers 16-byte aligned. Errors: INVALID_ARG, SHAPE,
 * ALIGNMENT, CUDA. */
int moe_combine_backward(const moe_desc_t* desc, const void* grad_out, const float* topk_weights,
                         const int32_t* slot_of, const void* expert_out, int64_t rows,
                         void* grad_expert_out, float* grad_weights, moe_stream_t stream);

/* Backward of dispatch with a BF16 payload (FP8 and NVFP4 taken as identity,
 * the straight-through reading): every pair's record carried the token's row,
 * so the gradient of that row is the sum of its pairs' gradient rows,
 *   grad_hidden[t] = bf16_rn( fp32 sum, ascending j, of grad_in[slot_of[t,j]] )
 * i.e. moe_combine (TOPK) with unit weights. grad_in bf16 [rows, H];
 * grad_hidden bf16 [N, H]. Errors: as moe_combine. */
int moe_dispatch_backward(const moe_desc_t* desc, const void* grad_in, int64_t rows,
                          const int32_t* slot_of, void* grad_hidden, moe_stream_t stream);

/* Backward of moe_combine_gather_ranks: every rank row the token's sum read
 * gets the token's gradient, grad_recv[send_head[t, r]] = grad_out[t] for each
 * r with send_head[t, r] in [0, recv_rows). grad_out bf16 [N, H]; grad_recv
 * bf16 [recv_rows, H]; only named rows are written. The backward of
 * moe_dispatch_ranks is moe_combine_gather_ranks itself. Errors: INVALID_ARG,
 * SHAPE, ALIGNMENT, CUDA. */
int moe_combine_gather_ranks_backward(const moe_desc_t* desc, const void* grad_out,
                                      const int32_t* send_head, void* grad_recv,
                                      int64_t recv_rows, moe_stream_t stream);

/* ---- tensor-major rank slots and padded-token mask ----------------------
 * The decode all-gather of the vLLM compare view ds-exp-2...ds-exp-ag packs
 * each rank's 2-4 tensors (top-k ids, weights, hidden payload, scales) into
 * one slot, one after the other at 16-byte-aligned offsets (moe_allgather.cu
 * "Host launcher", make_desc), and the gathered output of tensor i is every
 * rank's tensor i in rank order. Here the R ranks are regions of one GPU: the
 * tensors are [R][bytes[i]] (rank-major) and the slots [R][slot_bytes]. */
#define MOE_MAX_SLOT_TENSORS 4
typedef struct {
  int32_t num_tensors; /* 2..4 */
  int32_t num_ranks;   /* >= 1 */
  int64_t bytes[MOE_MAX_SLOT_TENSORS]; /* bytes of tensor i per rank, multiples of 16 */
} moe_slot_desc_t;

/* Host only. offsets[i] of tensor i inside a slot (num_tensors entries) and
 * the slot size. Errors: INVALID_ARG (NULL, num_tensors outside 2..4,
 * num_ranks < 1, negative size), ALIGNMENT (a size not a multiple of 16, as
 * make_desc rejects it). */
int moe_slot_layout(const moe_slot_desc_t* desc, int64_t* offsets, int64_t* slot_bytes);

/* Packs tensor i of rank r into slots[r] at offsets[i]. tensors is a host
 * array of num_tensors device pointers; all device pointers 16-byte aligned.
 * Errors: as moe_slot_layout, plus ALIGNMENT, CUDA. */
int moe_pack_slots(const moe_slot_desc_t* desc, const void* const* tensors, void* slots,
                   moe_stream_t stream);

/* The inverse: tensor i of rank r from slots[r] at offsets[i]. */
int moe_unpack_slots(const moe_slot_desc_t* desc, const void* slots, void* const* tensors,
                     moe_stream_t stream);

/* Padded tokens (vLLM all2all.py mask_topk_ids): topk_idx[t, :] = -1 for
 * every t >= *num_actual_tokens, where num_actual_tokens is a device int32
 * read by the kernel (a negative count masks every token), so a captured CUDA
 * graph stays valid as the count changes. topk_idx: device int32 [N, k].
 * Errors: INVALID_ARG, SHAPE, ALIGNMENT, CUDA. */
int moe_mask_topk_ids(int32_t* topk_idx, int32_t num_tokens, int32_t topk,
                      const int32_t* num_actual_tokens, moe_stream_t stream);

/* Host only: builds one record in host memory `record` (record_bytes bytes)
 * from host rows: ids_row int32 [k], w_row fp32 [k], payload_row
 * (payload_bytes, already in the out_kind format), scales_row (scale_bytes,
 * may be NULL when scale_bytes is 0). Padding is zeroed. Errors: INVALID_ARG,
 * SHAPE. */
int moe_pack_record(const moe_desc_t* desc, int32_t src_token, int32_t slot_j, int32_t expert,
                    const int32_t* ids_row, const float* w_row, const void* payload_row,
                    const void* scales_row, void* record);

/* Host only: the inverse of moe_pack_record. Any output pointer may be NULL to
 * skip that field. Errors: INVALID_ARG, SHAPE. */
int moe_unpack_record(const moe_desc_t* desc, const void* record, int32_t* src_token,
                      int32_t* slot_j, int32_t* expert, int32_t* ids_row, float* w_row,
                      void* payload_row, void* scales_row);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H */
