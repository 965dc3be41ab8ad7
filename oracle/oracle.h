/*
 * oracle.h -- plain, slow CPU oracle of MoE token dispatch and combine.
 *
 * TEST INFRASTRUCTURE ONLY. Only tests, the package smoke check and the
 * benchmark's CPU-baseline leg may load this code. The CUDA library never
 * includes, links or calls it, and this file includes nothing of the CUDA
 * library.
 *
 * Every routine computes the plain definition of one step, single-threaded,
 * in the precision the pages fix (fp32 accumulation, BF16 round-to-nearest-
 * even output; vLLM ds-exp-ag compare view, moe_reduce_scatter.cu, "bf16 <->
 * fp32 helpers") or in fp64 where it only bounds an error. Where the pages
 * leave a step open, the reading taken is written beside the routine.
 *
 * Integers are little-endian in records. Return value 0 = success, negative =
 * invalid argument.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Payload kinds: what a record carries in its payload segment. */
enum { ORACLE_BF16 = 0, ORACLE_FP8_E4M3_B128 = 1, ORACLE_NVFP4_B16 = 2, ORACLE_RAW = 3,
       ORACLE_FP8_E4M3_UE8M0 = 4 };

/* ---- number formats ---------------------------------------------------- */
float    oracle_bf16_to_f32(uint16_t b);
uint16_t oracle_f32_to_bf16(float f);     /* nearest, ties to even */
float    oracle_e4m3_value(uint8_t code);  /* OCP FP8 e4m3fn decode */
uint8_t  oracle_e4m3_encode(float x);      /* nearest finite, ties even, saturating */
float    oracle_e2m1_value(uint8_t code);  /* 4-bit FP4 e2m1 decode */
uint8_t  oracle_e2m1_encode(float x);      /* nearest, ties even, saturating */

/* ---- quantisers of one group of BF16 values ----------------------------- */
void oracle_fp8_group(const uint16_t* x, int n, uint8_t* q, float* scale);
void oracle_nvfp4_group(const uint16_t* x, int n, uint8_t* q_packed, uint8_t* scale);
void oracle_fp8_ue8m0_group(const uint16_t* x, int n, uint8_t* q, uint8_t* byte);

/* ---- record layout: out[7] = {record_bytes, off_ids, off_weights,
 *      off_payload, off_scales, payload_bytes, scale_bytes} ------------ */
int oracle_record_layout(int topk, int hidden, int in_kind, int out_kind,
                         int raw_payload_bytes, int raw_scale_bytes, int32_t* out);

/* ---- layout: counts, rank mask, scans, stable slot map ------------------ */
int oracle_layout(const int32_t* topk_idx, int num_tokens, int topk, int num_experts,
                  int num_ranks, int32_t* tokens_per_expert, int32_t* tokens_per_rank,
                  uint8_t* is_token_in_rank, int32_t* expert_offset, int32_t* rank_offset,
                  int32_t* slot_of, int32_t* src_of_slot);

/* ---- dispatch: quantise once per token, write one record per pair ------- */
int oracle_dispatch(const int32_t* topk_idx, const float* topk_weights,
                    const void* hidden, const void* scales, int num_tokens, int topk,
                    int hidden_size, int in_kind, int out_kind, int raw_payload_bytes,
                    int raw_scale_bytes, const int32_t* slot_of, uint8_t* records);

/* ---- identity expert: each record's payload back to BF16 rows ----------- */
int oracle_identity_expert(const uint8_t* records, int num_records, int topk,
                           int hidden_size, int out_kind, uint16_t* y);

/* ---- combine ------------------------------------------------------------- */
int oracle_combine_topk(const uint16_t* y, const float* topk_weights, const int32_t* slot_of,
                        int num_tokens, int topk, int hidden_size, uint16_t* out);
int oracle_combine_ranks(const uint16_t* partials, int num_ranks, int num_tokens,
                         int hidden_size, uint16_t* out);
int oracle_combine_topk_ranks(const uint16_t* y, const int32_t* topk_idx,
                              const float* topk_weights, const int32_t* slot_of,
                              int num_tokens, int topk, int num_experts, int num_ranks,
                              int hidden_size, uint16_t* out);
/* Combine + residual add + RMSNorm. mode 0 = top-k (y [P,H]), 1 = rank sum
 * (y = partials [R][N][H]), 2 = top-k grouped by rank. */
int oracle_combine_norm(int mode, const uint16_t* y, const int32_t* topk_idx,
                        const float* topk_weights, const int32_t* slot_of, int num_tokens,
                        int topk, int num_experts, int num_ranks, int hidden_size,
                        const uint16_t* residual, const uint16_t* gamma, float eps,
                        uint16_t* normed, uint16_t* residual_out);
/* One record per (token, destination rank) ([EP] intranode dispatch/combine). */
int oracle_rank_layout(const uint8_t* is_token_in_rank, const int32_t* tokens_per_expert,
                       int num_tokens, int num_ranks, int num_experts, int expert_alignment,
                       int32_t* send_head, int32_t* recv_src_idx, int32_t* recv_offset,
                       int32_t* recv_tokens_per_expert);
int oracle_dispatch_ranks(const int32_t* topk_idx, const float* topk_weights, const void* hidden,
                          const void* scales, int num_tokens, int topk, int num_experts,
                          int num_ranks, int hidden_size, int in_kind, int out_kind,
                          int raw_payload_bytes, int raw_scale_bytes, const int32_t* send_head,
                          uint8_t* records);
int oracle_combine_gather_ranks(const uint16_t* recv_out, const int32_t* send_head,
                                int num_tokens, int num_ranks, int hidden_size, uint16_t* out);
/* Fixed-capacity, expert-major receive buffers ([EP] low-latency dispatch). */
int oracle_ll_layout(const int32_t* topk_idx, int num_tokens, int topk, int num_experts,
                     int num_ranks, int max_tokens_per_rank, int32_t* ll_slot_of,
                     int32_t* src_info, int64_t* layout_range, int32_t* recv_count);
int oracle_dispatch_ll(const void* hidden, const void* scales, int num_tokens, int topk,
                       int hidden_size, int in_kind, int out_kind, int raw_payload_bytes,
                       int raw_scale_bytes, const int32_t* ll_slot_of, int64_t rows,
                       uint8_t* x_out, uint8_t* scales_out);
/* Backward ([EP] README, model training example: the backward of combine is
 * a dispatch through the cached handle, the backward of dispatch a combine). */
int oracle_combine_backward(const uint16_t* grad_out, const float* topk_weights,
                            const int32_t* slot_of, const uint16_t* y, int64_t rows,
                            int num_tokens, int topk, int hidden_size, uint16_t* grad_y,
                            float* grad_w);
int oracle_dispatch_backward(const uint16_t* grad_in, const int32_t* slot_of, int num_tokens,
                             int topk, int hidden_size, uint16_t* grad_hidden);
int oracle_gather_ranks_backward(const uint16_t* grad_out, const int32_t* send_head,
                                 int num_tokens, int num_ranks, int hidden_size, int64_t rows,
                                 uint16_t* grad_recv);
/* Rank slots of the decode all-gather ([AG] make_desc) and the padded-token
 * mask ([AG] mask_topk_ids). */
int oracle_slot_layout(int num_tensors, const int64_t* bytes, int64_t* offsets, int64_t* slot_bytes);
int oracle_pack_slots(int num_tensors, int num_ranks, const int64_t* bytes,
                      const uint8_t* const* tensors, uint8_t* slots);
int oracle_unpack_slots(int num_tensors, int num_ranks, const int64_t* bytes,
                        const uint8_t* slots, uint8_t* const* tensors);
void oracle_mask_topk_ids(int32_t* topk_idx, int num_tokens, int topk, int num_actual_tokens);
/* fp64 references, used only to bound the error of the fp32 routines */
int oracle_combine_topk_f64(const uint16_t* y, const float* topk_weights,
                            const int32_t* slot_of, int num_tokens, int topk,
                            int hidden_size, double* out);

#ifdef __cplusplus
}
#endif
#endif
