/*
 * oracle.c -- plain, slow CPU oracle of MoE token dispatch and combine.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by tests, the smoke check and the CPU
 * baseline of the benchmark, never by the CUDA library. Built with
 * -O2 -ffp-contract=off and without fast-math, so every float operation
 * below is one IEEE-754 operation in the order written.
 *
 * Sources, by page:
 *  [AG]  vLLM compare view woosuk/ds-exp-2...woosuk/ds-exp-ag:
 *        moe_allgather.cu "Host launcher" (tensors packed at 16-byte aligned
 *        offsets, make_desc); moe_reduce_scatter.cu "bf16 <-> fp32 helpers"
 *        and "Lamport reduce-scatter kernel" phase 3 (fp32 sum over ranks in
 *        ascending order, one BF16 rounding); all2all.py mask_topk_ids
 *        (-1 marks a token with no expert); bench_moe_allgather.py (decode
 *        payload: 3584 NVFP4 bytes + 448 e4m3 scales per token).
 *  [PR]  vLLM PR "Eliminate staging from NCCL symmetric reduce-scatter",
 *        Summary/Implementation (top-k reduction written straight into the
 *        buffer the reduce-scatter sums).
 *  [EP]  DeepEP repository: csrc/deep_ep.cpp Buffer::get_dispatch_layout
 *        (per-rank and per-expert counts, is_token_in_rank),
 *        Buffer::low_latency_dispatch (FP8 cast with fp32 scales per 128
 *        channels; E % R == 0, E/R local experts per rank),
 *        Buffer::low_latency_combine (top-k weighted reduction back to token
 *        order); csrc/config.hpp LowLatencyLayout (message = int4 header +
 *        payload + scales).
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ======================================================================== */
/* Number formats                                                            */
/* ======================================================================== */

float oracle_bf16_to_f32(uint16_t b) {
  /* BF16 is the upper half of an fp32 bit pattern. */
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* Nearest BF16 value to f; on a tie, the one with an even last mantissa bit
 * (the rounding of __float2bfloat16 in [AG] "bf16 <-> fp32 helpers"). The two
 * candidates are f truncated toward zero and the next BF16 away from zero;
 * distances are exact in double. */
uint16_t oracle_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if (isnan(f)) return (uint16_t)((u >> 16) | 0x0040u);
  if (isinf(f)) return (uint16_t)(u >> 16);
  uint16_t lo = (uint16_t)(u >> 16);
  uint16_t hi = (uint16_t)(lo + 1u);
  double vlo = fabs((double)oracle_bf16_to_f32(lo));
  double vhi = ((hi & 0x7fffu) == 0x7f80u) ? ldexp(1.0, 128) /* overflow step */
                                           : fabs((double)oracle_bf16_to_f32(hi));
  double af = fabs((double)f);
  double dlo = af - vlo, dhi = vhi - af;
  if (dlo < dhi) return lo;
  if (dhi < dlo) return hi;
  return (lo & 1u) ? hi : lo;
}

/* OCP FP8 e4m3fn: sign, 4 exponent bits (bias 7), 3 mantissa bits, no
 * infinities, S.1111.111 is NaN. Exponent field 0 is subnormal: m * 2^-9. */
float oracle_e4m3_value(uint8_t code) {
  int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
  if (e == 15 && m == 7) return NAN;
  float v = (e == 0) ? ldexpf((float)m, -9) : ldexpf((float)(8 + m), e - 10);
  return s ? -v : v;
}

/* The finite e4m3 value nearest to x (ties to the even code), sign kept;
 * anything beyond the largest finite value 448 becomes +-448 (saturation). */
uint8_t oracle_e4m3_encode(float x) {
  uint8_t sign = signbit(x) ? 0x80 : 0x00;
  if (isnan(x)) return (uint8_t)(sign | 0x7f);
  double ax = fabs((double)x);
  if (ax >= 448.0) return (uint8_t)(sign | 0x7e);
  int best = 0;
  double bestd = INFINITY;
  for (int c = 0; c <= 0x7e; ++c) {
    double d = fabs(ax - (double)oracle_e4m3_value((uint8_t)c));
    if (d < bestd || (d == bestd && (c & 1) == 0 && (best & 1) == 1)) {
      best = c;
      bestd = d;
    }
  }
  return (uint8_t)(sign | best);
}

/* FP4 e2m1: sign bit 3, magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6} for codes 0..7. */
static const float kE2M1[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};

float oracle_e2m1_value(uint8_t code) {
  float v = kE2M1[code & 7];
  return (code & 8) ? -v : v;
}

uint8_t oracle_e2m1_encode(float x) {
  uint8_t sign = signbit(x) ? 8 : 0;
  double ax = fabs((double)x);
  if (ax >= 6.0) return (uint8_t)(sign | 7);
  int best = 0;
  double bestd = INFINITY;
  for (int c = 0; c < 8; ++c) {
    double d = fabs(ax - (double)kE2M1[c]);
    if (d < bestd || (d == bestd && (c & 1) == 0 && (best & 1) == 1)) {
      best = c;
      bestd = d;
    }
  }
  return (uint8_t)(sign | best);
}

/* ======================================================================== */
/* Quantisers                                                                */
/* ======================================================================== */

/* FP8 e4m3 with one fp32 scale per group of 128 channels ([EP]
 * low_latency_dispatch "ptp128c" cast; the pages give no formula). Reading:
 *   amax = max |x_i|;  a = max(amax, 1e-4);  scale = a / 448;  inv = 448 / a;
 *   q_i = e4m3(x_i * inv)  (round to nearest even, saturating).
 * Dequantised value: e4m3_value(q_i) * scale. */
void oracle_fp8_group(const uint16_t* x, int n, uint8_t* q, float* scale) {
  float amax = 0.0f;
  for (int i = 0; i < n; ++i) {
    float v = fabsf(oracle_bf16_to_f32(x[i]));
    if (v > amax) amax = v;
  }
  float a = (amax > 1e-4f) ? amax : 1e-4f;
  float s = a / 448.0f;
  float inv = 448.0f / a;
  for (int i = 0; i < n; ++i) q[i] = oracle_e4m3_encode(oracle_bf16_to_f32(x[i]) * inv);
  *scale = s;
}

/* FP8 e4m3 per 128 channels with a power-of-two scale kept as one UE8M0
 * byte ([EP] Buffer::low_latency_dispatch: use_ue8m0 requires round_scale,
 * and the scales become int32 [E_l, H/512, R * maxT] -- one byte per
 * 128-channel group, four groups to an int). The pages give no formula.
 * Reading: the scale is rounded up to a power of two, so nothing saturates:
 *   a = max(amax, 1e-4);  v = a / 448 (IEEE fp32);
 *   e = the least integer with 2^e >= v;
 *   q_i = e4m3(x_i * 2^-e)   (multiplying by a power of two is exact);
 *   byte = e + 127           (UE8M0 stores the biased exponent: 2^(byte-127)). */
void oracle_fp8_ue8m0_group(const uint16_t* x, int n, uint8_t* q, uint8_t* byte) {
  float amax = 0.0f;
  for (int i = 0; i < n; ++i) {
    float v = fabsf(oracle_bf16_to_f32(x[i]));
    if (v > amax) amax = v;
  }
  float a = (amax > 1e-4f) ? amax : 1e-4f;
  float v = a / 448.0f;
  int ex;
  double m = frexp((double)v, &ex); /* v = m * 2^ex, m in [0.5, 1) */
  int e = (m == 0.5) ? ex - 1 : ex;
  float inv = ldexpf(1.0f, -e);
  for (int i = 0; i < n; ++i) q[i] = oracle_e4m3_encode(oracle_bf16_to_f32(x[i]) * inv);
  *byte = (uint8_t)(e + 127);
}

/* NVFP4: FP4 e2m1 values with one e4m3 scale byte per group of 16 ([AG]
 * decode payload: 3584 packed bytes + 448 scale bytes for hidden 7168). The
 * pages give no formula and no global scale. Reading:
 *   amax = max |x_i|;  sc = e4m3(amax / 6);  d = e4m3_value(sc);
 *   q_i = 0 if d == 0, else e2m1(x_i / d);
 *   byte i holds element 2i in its low nibble and 2i+1 in its high nibble. */
void oracle_nvfp4_group(const uint16_t* x, int n, uint8_t* q_packed, uint8_t* scale) {
  float amax = 0.0f;
  for (int i = 0; i < n; ++i) {
    float v = fabsf(oracle_bf16_to_f32(x[i]));
    if (v > amax) amax = v;
  }
  uint8_t sc = oracle_e4m3_encode(amax / 6.0f);
  float d = oracle_e4m3_value(sc);
  for (int i = 0; i < n; i += 2) {
    uint8_t c0 = 0, c1 = 0;
    if (d != 0.0f) {
      c0 = oracle_e2m1_encode(oracle_bf16_to_f32(x[i]) / d);
      c1 = oracle_e2m1_encode(oracle_bf16_to_f32(x[i + 1]) / d);
    }
    q_packed[i / 2] = (uint8_t)(c0 | (c1 << 4));
  }
  *scale = sc;
}

/* ======================================================================== */
/* Record layout                                                             */
/* ======================================================================== */

static int pad16(int x) { return (x + 15) / 16 * 16; }

/* One record per (token, top-k slot) pair. Segments, each starting at a
 * 16-byte boundary ([AG] make_desc packs tensors at 16-byte aligned
 * offsets; [EP] LowLatencyLayout: an int4 header, then payload, then
 * scales), padding bytes zero:
 *   header  16 bytes: int32 src_token, int32 j, int32 expert, int32 0
 *   ids     the token's whole top-k id row (int32 x k)
 *   weights the token's fp32 weight row (fp32 x k)
 *   payload BF16 row | FP8 bytes | packed NVFP4 | raw bytes
 *   scales  none | fp32 per 128 | e4m3 byte per 16 | raw bytes */
int oracle_record_layout(int topk, int hidden, int in_kind, int out_kind,
                         int raw_payload_bytes, int raw_scale_bytes, int32_t* out) {
  int pb, sb;
  if (topk < 1 || hidden < 0) return -1;
  if (out_kind == ORACLE_BF16 && in_kind == ORACLE_BF16) {
    pb = hidden * 2;
    sb = 0;
  } else if (out_kind == ORACLE_FP8_E4M3_B128 && in_kind == ORACLE_BF16) {
    if (hidden % 128) return -1;
    pb = hidden;
    sb = hidden / 128 * 4;
  } else if (out_kind == ORACLE_NVFP4_B16 && in_kind == ORACLE_BF16) {
    if (hidden % 16) return -1;
    pb = hidden / 2;
    sb = hidden / 16;
  } else if (out_kind == ORACLE_FP8_E4M3_UE8M0 && in_kind == ORACLE_BF16) {
    if (hidden % 128) return -1;
    pb = hidden;
    sb = hidden / 128;
  } else if (out_kind == ORACLE_RAW && in_kind == ORACLE_RAW) {
    if (raw_payload_bytes < 0 || raw_scale_bytes < 0) return -1;
    pb = raw_payload_bytes;
    sb = raw_scale_bytes;
  } else {
    return -1;
  }
  int off_ids = 16;
  int off_w = off_ids + pad16(4 * topk);
  int off_p = off_w + pad16(4 * topk);
  int off_s = off_p + pad16(pb);
  out[0] = off_s + pad16(sb);
  out[1] = off_ids;
  out[2] = off_w;
  out[3] = off_p;
  out[4] = off_s;
  out[5] = pb;
  out[6] = sb;
  return 0;
}

/* ======================================================================== */
/* Layout ([EP] get_dispatch_layout plus the slot map)                       */
/* ======================================================================== */

/* Expert e lives on rank e / (E/R): contiguous blocks of E/R local experts
 * ([EP] num_local_experts = num_experts / num_ranks). An id of -1 means "no
 * expert" ([AG] mask_topk_ids) and counts nowhere; any other id outside
 * [0, E) is an error.
 *   tokens_per_expert[e]   number of pairs (t, j) routed to e
 *   is_token_in_rank[t, r] 1 if some pair of token t goes to rank r
 *   tokens_per_rank[r]     number of tokens t with is_token_in_rank[t, r]
 *   expert_offset[e]       exclusive prefix sum of tokens_per_expert (E+1)
 *   rank_offset[r]         expert_offset[r * E/R] (R+1)
 *   slot_of[t, j]          expert_offset[e] + number of earlier pairs (in
 *                          (t, j) order) with the same expert; -1 if e < 0
 *   src_of_slot[s]         t * k + j of the pair in slot s; -1 past the
 *                          last used slot (array length N * k)
 * The order inside an expert's region is ascending (t, j): a stable counting
 * sort of the pairs by expert (the pages do not fix this order). */
int oracle_layout(const int32_t* topk_idx, int num_tokens, int topk, int num_experts,
                  int num_ranks, int32_t* tokens_per_expert, int32_t* tokens_per_rank,
                  uint8_t* is_token_in_rank, int32_t* expert_offset, int32_t* rank_offset,
                  int32_t* slot_of, int32_t* src_of_slot) {
  if (num_tokens < 0 || topk < 1 || num_experts < 1 || num_ranks < 1) return -1;
  if (num_experts % num_ranks != 0) return -1;
  const int per_rank = num_experts / num_ranks;
  const long pairs = (long)num_tokens * topk;
  for (long p = 0; p < pairs; ++p)
    if (topk_idx[p] < -1 || topk_idx[p] >= num_experts) return -1;

  for (int e = 0; e < num_experts; ++e) tokens_per_expert[e] = 0;
  for (int r = 0; r < num_ranks; ++r) tokens_per_rank[r] = 0;
  for (int t = 0; t < num_tokens; ++t) {
    uint8_t* row = is_token_in_rank + (long)t * num_ranks;
    for (int r = 0; r < num_ranks; ++r) row[r] = 0;
    for (int j = 0; j < topk; ++j) {
      int e = topk_idx[(long)t * topk + j];
      if (e < 0) continue;
      tokens_per_expert[e] += 1;
      row[e / per_rank] = 1;
    }
    for (int r = 0; r < num_ranks; ++r) tokens_per_rank[r] += row[r];
  }

  expert_offset[0] = 0;
  for (int e = 0; e < num_experts; ++e) expert_offset[e + 1] = expert_offset[e] + tokens_per_expert[e];
  for (int r = 0; r < num_ranks; ++r) rank_offset[r] = expert_offset[r * per_rank];
  rank_offset[num_ranks] = expert_offset[num_experts];

  int32_t* cursor = (int32_t*)malloc(sizeof(int32_t) * (size_t)num_experts);
  if (!cursor) return -2;
  for (int e = 0; e < num_experts; ++e) cursor[e] = expert_offset[e];
  if (src_of_slot)
    for (long s = 0; s < pairs; ++s) src_of_slot[s] = -1;
  for (int t = 0; t < num_tokens; ++t) {
    for (int j = 0; j < topk; ++j) {
      long p = (long)t * topk + j;
      int e = topk_idx[p];
      if (e < 0) {
        slot_of[p] = -1;
        continue;
      }
      int s = cursor[e]++;
      slot_of[p] = s;
      if (src_of_slot) src_of_slot[s] = (int32_t)p;
    }
  }
  free(cursor);
  return 0;
}

/* ======================================================================== */
/* Dispatch                                                                  */
/* ======================================================================== */

/* The payload of one token is computed once; every valid pair (t, j) then
 * gets its own record at records + slot_of[t, j] * record_bytes. */
int oracle_dispatch(const int32_t* topk_idx, const float* topk_weights,
                    const void* hidden, const void* scales, int num_tokens, int topk,
                    int hidden_size, int in_kind, int out_kind, int raw_payload_bytes,
                    int raw_scale_bytes, const int32_t* slot_of, uint8_t* records) {
  int32_t lay[7];
  if (oracle_record_layout(topk, hidden_size, in_kind, out_kind, raw_payload_bytes,
                           raw_scale_bytes, lay) != 0)
    return -1;
  const int S = lay[0], off_ids = lay[1], off_w = lay[2], off_p = lay[3], off_s = lay[4];
  const int pb = lay[5], sb = lay[6];
  uint8_t* pay = (uint8_t*)malloc((size_t)pb + 1);
  uint8_t* sca = (uint8_t*)malloc((size_t)sb + 1);
  if (!pay || !sca) {
    free(pay);
    free(sca);
    return -2;
  }
  for (int t = 0; t < num_tokens; ++t) {
    /* this token's payload and scales */
    if (out_kind == ORACLE_BF16) {
      memcpy(pay, (const uint8_t*)hidden + (size_t)t * hidden_size * 2, (size_t)pb);
    } else if (out_kind == ORACLE_FP8_E4M3_B128) {
      const uint16_t* x = (const uint16_t*)hidden + (size_t)t * hidden_size;
      for (int g = 0; g < hidden_size / 128; ++g) {
        float sc;
        oracle_fp8_group(x + g * 128, 128, pay + g * 128, &sc);
        memcpy(sca + g * 4, &sc, 4);
      }
    } else if (out_kind == ORACLE_NVFP4_B16) {
      const uint16_t* x = (const uint16_t*)hidden + (size_t)t * hidden_size;
      for (int g = 0; g < hidden_size / 16; ++g) oracle_nvfp4_group(x + g * 16, 16, pay + g * 8, sca + g);
    } else if (out_kind == ORACLE_FP8_E4M3_UE8M0) {
      const uint16_t* x = (const uint16_t*)hidden + (size_t)t * hidden_size;
      for (int g = 0; g < hidden_size / 128; ++g)
        oracle_fp8_ue8m0_group(x + g * 128, 128, pay + g * 128, sca + g);
    } else { /* RAW: opaque bytes, copied as they are */
      memcpy(pay, (const uint8_t*)hidden + (size_t)t * pb, (size_t)pb);
      if (sb) memcpy(sca, (const uint8_t*)scales + (size_t)t * sb, (size_t)sb);
    }
    for (int j = 0; j < topk; ++j) {
      long p = (long)t * topk + j;
      int s = slot_of[p];
      if (s < 0) continue;
      uint8_t* rec = records + (size_t)s * S;
      memset(rec, 0, (size_t)S);
      int32_t hdr[4] = {t, j, topk_idx[p], 0};
      memcpy(rec, hdr, 16);
      memcpy(rec + off_ids, topk_idx + (long)t * topk, (size_t)topk * 4);
      memcpy(rec + off_w, topk_weights + (long)t * topk, (size_t)topk * 4);
      memcpy(rec + off_p, pay, (size_t)pb);
      if (sb) memcpy(rec + off_s, sca, (size_t)sb);
    }
  }
  free(pay);
  free(sca);
  return 0;
}

/* An expert that returns its input: the record's payload turned back into a
 * BF16 row (FP8: e4m3_value(q) * scale; NVFP4: e2m1_value(q) * e4m3_value(sc);
 * each product in fp32, then rounded to BF16). */
int oracle_identity_expert(const uint8_t* records, int num_records, int topk,
                           int hidden_size, int out_kind, uint16_t* y) {
  int32_t lay[7];
  if (oracle_record_layout(topk, hidden_size, ORACLE_BF16, out_kind, 0, 0, lay) != 0) return -1;
  const int S = lay[0], off_p = lay[3], off_s = lay[4];
  for (int s = 0; s < num_records; ++s) {
    const uint8_t* rec = records + (size_t)s * S;
    uint16_t* row = y + (size_t)s * hidden_size;
    for (int h = 0; h < hidden_size; ++h) {
      if (out_kind == ORACLE_BF16) {
        memcpy(&row[h], rec + off_p + 2 * h, 2);
      } else if (out_kind == ORACLE_FP8_E4M3_B128) {
        float sc;
        memcpy(&sc, rec + off_s + 4 * (h / 128), 4);
        row[h] = oracle_f32_to_bf16(oracle_e4m3_value(rec[off_p + h]) * sc);
      } else if (out_kind == ORACLE_FP8_E4M3_UE8M0) {
        int e = (int)rec[off_s + h / 128] - 127;
        row[h] = oracle_f32_to_bf16(ldexpf(oracle_e4m3_value(rec[off_p + h]), e));
      } else {
        uint8_t b = rec[off_p + h / 2];
        uint8_t c = (h & 1) ? (uint8_t)(b >> 4) : (uint8_t)(b & 15);
        row[h] = oracle_f32_to_bf16(oracle_e2m1_value(c) * oracle_e4m3_value(rec[off_s + h / 16]));
      }
    }
  }
  return 0;
}

/* ======================================================================== */
/* Combine                                                                   */
/* ======================================================================== */

/* Top-k weighted reduction back to token order ([EP] low_latency_combine):
 *   out[t, h] = bf16( fma chain over j = 0..k-1 with slot_of[t, j] >= 0 of
 *                     w[t, j] * y[slot_of[t, j], h], starting from +0 )
 * One fp32 accumulator per element, ascending j, one fused multiply-add per
 * term, one BF16 rounding at the end. (fp32 accumulation and the BF16
 * rounding follow [AG]; ascending j and the fused multiply-add are the
 * reading taken where the pages are silent.) */
int oracle_combine_topk(const uint16_t* y, const float* topk_weights, const int32_t* slot_of,
                        int num_tokens, int topk, int hidden_size, uint16_t* out) {
  float* acc = (float*)malloc(sizeof(float) * (size_t)(hidden_size > 0 ? hidden_size : 1));
  if (!acc) return -2;
  for (int t = 0; t < num_tokens; ++t) {
    for (int h = 0; h < hidden_size; ++h) acc[h] = 0.0f;
    for (int j = 0; j < topk; ++j) {
      long p = (long)t * topk + j;
      int s = slot_of[p];
      if (s < 0) continue;
      float w = topk_weights[p];
      const uint16_t* row = y + (size_t)s * hidden_size;
      for (int h = 0; h < hidden_size; ++h) acc[h] = fmaf(w, oracle_bf16_to_f32(row[h]), acc[h]);
    }
    for (int h = 0; h < hidden_size; ++h) out[(size_t)t * hidden_size + h] = oracle_f32_to_bf16(acc[h]);
  }
  free(acc);
  return 0;
}

/* The cross-rank sum a reduce-scatter performs ([AG] "Lamport reduce-scatter
 * kernel" phase 3): partials is [R][N][H] BF16; for every row n and column h,
 *   out[n, h] = bf16( ((0 + P_0[n,h]) + P_1[n,h]) + ... + P_{R-1}[n,h] )
 * in fp32, ranks in ascending order. Rank q's reduce-scatter output is rows
 * [q*N/R, (q+1)*N/R) of out; N % R == 0 as the page requires. */
int oracle_combine_ranks(const uint16_t* partials, int num_ranks, int num_tokens,
                         int hidden_size, uint16_t* out) {
  if (num_ranks < 1 || num_tokens % num_ranks) return -1;
  for (long n = 0; n < num_tokens; ++n) {
    for (int h = 0; h < hidden_size; ++h) {
      float acc = 0.0f;
      for (int r = 0; r < num_ranks; ++r)
        acc = acc + oracle_bf16_to_f32(partials[((size_t)r * num_tokens + n) * hidden_size + h]);
      out[n * hidden_size + h] = oracle_f32_to_bf16(acc);
    }
  }
  return 0;
}

/* Top-k reduction written straight into the rank sum ([PR] Implementation):
 * for each rank r the partial is the fp32 fma chain (ascending j, from +0)
 * over the pairs whose expert lives on rank r; the partials are then summed
 * in fp32 in ascending r (from +0) and rounded to BF16 once. Reading: the
 * partials stay fp32 (one rounding in all), since no rank boundary is
 * crossed on one GPU. N % R == 0 so that rank q owns rows [qN/R, (q+1)N/R). */
int oracle_combine_topk_ranks(const uint16_t* y, const int32_t* topk_idx,
                              const float* topk_weights, const int32_t* slot_of,
                              int num_tokens, int topk, int num_experts, int num_ranks,
                              int hidden_size, uint16_t* out) {
  if (num_ranks < 1 || num_experts % num_ranks || num_tokens % num_ranks) return -1;
  const int per_rank = num_experts / num_ranks;
  size_t hs = (size_t)(hidden_size > 0 ? hidden_size : 1);
  float* total = (float*)malloc(sizeof(float) * hs);
  float* part = (float*)malloc(sizeof(float) * hs);
  if (!total || !part) {
    free(total);
    free(part);
    return -2;
  }
  for (int t = 0; t < num_tokens; ++t) {
    for (int h = 0; h < hidden_size; ++h) total[h] = 0.0f;
    for (int r = 0; r < num_ranks; ++r) {
      for (int h = 0; h < hidden_size; ++h) part[h] = 0.0f;
      for (int j = 0; j < topk; ++j) {
        long p = (long)t * topk + j;
        int s = slot_of[p];
        if (s < 0 || topk_idx[p] / per_rank != r) continue;
        float w = topk_weights[p];
        const uint16_t* row = y + (size_t)s * hidden_size;
        for (int h = 0; h < hidden_size; ++h) part[h] = fmaf(w, oracle_bf16_to_f32(row[h]), part[h]);
      }
      for (int h = 0; h < hidden_size; ++h) total[h] = total[h] + part[h];
    }
    for (int h = 0; h < hidden_size; ++h) out[(size_t)t * hidden_size + h] = oracle_f32_to_bf16(total[h]);
  }
  free(total);
  free(part);
  return 0;
}

int oracle_combine_topk_f64(const uint16_t* y, const float* topk_weights,
                            const int32_t* slot_of, int num_tokens, int topk,
                            int hidden_size, double* out) {
  for (int t = 0; t < num_tokens; ++t) {
    double* o = out + (size_t)t * hidden_size;
    for (int h = 0; h < hidden_size; ++h) o[h] = 0.0;
    for (int j = 0; j < topk; ++j) {
      long p = (long)t * topk + j;
      int s = slot_of[p];
      if (s < 0) continue;
      double w = (double)topk_weights[p];
      const uint16_t* row = y + (size_t)s * hidden_size;
      for (int h = 0; h < hidden_size; ++h) o[h] += w * (double)oracle_bf16_to_f32(row[h]);
    }
  }
  return 0;
}

/* Combine fused with the residual add and RMSNorm ([AG] moe_rs_fused.cu:
 * reduce-scatter sum in fp32, add the residual, RMSNorm over the row;
 * test_rs_fused.py rms_norm_ref: x * rsqrt(mean(x^2) + eps) * gamma in fp32).
 * For each token t:
 *   s[h]     = the mode's combine in fp32 before its final rounding, with the
 *              same operation order as oracle_combine_topk / _ranks /
 *              _topk_ranks
 *   x[h]     = s[h] + residual[t,h]                      (fp32 add)
 *   residual_out[t,h] = bf16(x[h])
 *   ms       = (sum over h of x[h]^2) / H                (fp64)
 *   r        = fp32(1 / sqrt(ms + eps))                  (fp64, rounded once)
 *   normed[t,h] = bf16((x[h] * r) * gamma[h])            (two fp32 products)
 * Reading: the pages sum the squares in fp32 in a tree order and use rsqrtf;
 * the oracle takes the exact-as-fp64 mean and one rounding of the scale, so
 * the normed output agrees with them only within rounding. */
int oracle_combine_norm(int mode, const uint16_t* y, const int32_t* topk_idx,
                        const float* topk_weights, const int32_t* slot_of, int num_tokens,
                        int topk, int num_experts, int num_ranks, int hidden_size,
                        const uint16_t* residual, const uint16_t* gamma, float eps,
                        uint16_t* normed, uint16_t* residual_out) {
  if (mode < 0 || mode > 2 || num_ranks < 1 || hidden_size < 1) return -1;
  if (mode != 0 && (num_tokens % num_ranks)) return -1;
  if (mode == 2 && num_experts % num_ranks) return -1;
  const int per_rank = mode == 2 ? num_experts / num_ranks : 1;
  const size_t hs = (size_t)hidden_size;
  float* x = (float*)malloc(sizeof(float) * hs);
  float* part = (float*)malloc(sizeof(float) * hs);
  if (!x || !part) {
    free(x);
    free(part);
    return -2;
  }
  for (int t = 0; t < num_tokens; ++t) {
    for (int h = 0; h < hidden_size; ++h) x[h] = 0.0f;
    if (mode == 0) {
      for (int j = 0; j < topk; ++j) {
        long p = (long)t * topk + j;
        int s = slot_of[p];
        if (s < 0) continue;
        float w = topk_weights[p];
        const uint16_t* row = y + (size_t)s * hs;
        for (int h = 0; h < hidden_size; ++h) x[h] = fmaf(w, oracle_bf16_to_f32(row[h]), x[h]);
      }
    } else if (mode == 1) {
      for (int r = 0; r < num_ranks; ++r)
        for (int h = 0; h < hidden_size; ++h)
          x[h] = x[h] + oracle_bf16_to_f32(y[((size_t)r * num_tokens + t) * hs + h]);
    } else {
      for (int r = 0; r < num_ranks; ++r) {
        for (int h = 0; h < hidden_size; ++h) part[h] = 0.0f;
        for (int j = 0; j < topk; ++j) {
          long p = (long)t * topk + j;
          int s = slot_of[p];
          if (s < 0 || topk_idx[p] / per_rank != r) continue;
          float w = topk_weights[p];
          const uint16_t* row = y + (size_t)s * hs;
          for (int h = 0; h < hidden_size; ++h) part[h] = fmaf(w, oracle_bf16_to_f32(row[h]), part[h]);
        }
        for (int h = 0; h < hidden_size; ++h) x[h] = x[h] + part[h];
      }
    }
    double sumsq = 0.0;
    for (int h = 0; h < hidden_size; ++h) {
      x[h] = x[h] + oracle_bf16_to_f32(residual[(size_t)t * hs + h]);
      residual_out[(size_t)t * hs + h] = oracle_f32_to_bf16(x[h]);
      sumsq += (double)x[h] * (double)x[h];
    }
    float r = (float)(1.0 / sqrt(sumsq / hidden_size + (double)eps));
    for (int h = 0; h < hidden_size; ++h)
      normed[(size_t)t * hs + h] = oracle_f32_to_bf16((x[h] * r) * oracle_bf16_to_f32(gamma[h]));
  }
  free(x);
  free(part);
  return 0;
}

/* ======================================================================== */
/* Rank slots and padded tokens                                              */
/* ======================================================================== */

/* [AG] moe_allgather.cu make_desc: a cursor walks the tensors in order; each
 * tensor starts at the cursor rounded up to 16 and must have a byte size that
 * is a multiple of 16; the slot is the final cursor. */
int oracle_slot_layout(int num_tensors, const int64_t* bytes, int64_t* offsets, int64_t* slot_bytes) {
  if (num_tensors < 2 || num_tensors > 4) return -1;
  int64_t cursor = 0;
  for (int i = 0; i < num_tensors; ++i) {
    if (bytes[i] < 0 || bytes[i] % 16) return -1;
    cursor = (cursor + 15) / 16 * 16;
    offsets[i] = cursor;
    cursor += bytes[i];
  }
  *slot_bytes = cursor;
  return 0;
}

/* Slot r holds tensor i of rank r (bytes[i] bytes at tensor + r*bytes[i]) at
 * offsets[i]; the gathered tensor i is all ranks' pieces in rank order. */
int oracle_pack_slots(int num_tensors, int num_ranks, const int64_t* bytes,
                      const uint8_t* const* tensors, uint8_t* slots) {
  int64_t off[4], sb;
  if (oracle_slot_layout(num_tensors, bytes, off, &sb) != 0 || num_ranks < 1) return -1;
  for (int r = 0; r < num_ranks; ++r)
    for (int i = 0; i < num_tensors; ++i)
      for (int64_t b = 0; b < bytes[i]; ++b)
        slots[(size_t)r * sb + off[i] + b] = tensors[i][(size_t)r * bytes[i] + b];
  return 0;
}

int oracle_unpack_slots(int num_tensors, int num_ranks, const int64_t* bytes,
                        const uint8_t* slots, uint8_t* const* tensors) {
  int64_t off[4], sb;
  if (oracle_slot_layout(num_tensors, bytes, off, &sb) != 0 || num_ranks < 1) return -1;
  for (int r = 0; r < num_ranks; ++r)
    for (int i = 0; i < num_tensors; ++i)
      for (int64_t b = 0; b < bytes[i]; ++b)
        tensors[i][(size_t)r * bytes[i] + b] = slots[(size_t)r * sb + off[i] + b];
  return 0;
}

/* [AG] all2all.py mask_topk_ids: every token t >= num_actual_tokens gets -1
 * in each of its k ids. */
void oracle_mask_topk_ids(int32_t* topk_idx, int num_tokens, int topk, int num_actual_tokens) {
  for (int t = 0; t < num_tokens; ++t)
    if (t >= num_actual_tokens)
      for (int j = 0; j < topk; ++j) topk_idx[(long)t * topk + j] = -1;
}

/* ======================================================================== */
/* One record per (token, destination rank)                                  */
/* ======================================================================== */

/* [EP] Buffer::intranode_dispatch: rank r receives every token t with
 * is_token_in_rank[t, r], here in ascending t (virtual source ranks own
 * contiguous token ranges). recv_offset is the exclusive prefix sum of the
 * per-rank token counts; send_head[t, r] is the token's receive slot or -1;
 * recv_src_idx[s] the token in slot s (-1 past the last, N*R entries); the
 * per-expert counts are rounded up to expert_alignment. */
int oracle_rank_layout(const uint8_t* is_token_in_rank, const int32_t* tokens_per_expert,
                       int num_tokens, int num_ranks, int num_experts, int expert_alignment,
                       int32_t* send_head, int32_t* recv_src_idx, int32_t* recv_offset,
                       int32_t* recv_tokens_per_expert) {
  if (num_tokens < 0 || num_ranks < 1 || num_experts < 1 || expert_alignment < 1) return -1;
  int run = 0;
  for (int r = 0; r < num_ranks; ++r) {
    recv_offset[r] = run;
    for (int t = 0; t < num_tokens; ++t) run += is_token_in_rank[(long)t * num_ranks + r] ? 1 : 0;
  }
  recv_offset[num_ranks] = run;
  if (recv_src_idx)
    for (long s = 0; s < (long)num_tokens * num_ranks; ++s) recv_src_idx[s] = -1;
  for (int r = 0; r < num_ranks; ++r) {
    int cursor = recv_offset[r];
    for (int t = 0; t < num_tokens; ++t) {
      if (is_token_in_rank[(long)t * num_ranks + r]) {
        send_head[(long)t * num_ranks + r] = cursor;
        if (recv_src_idx) recv_src_idx[cursor] = t;
        ++cursor;
      } else {
        send_head[(long)t * num_ranks + r] = -1;
      }
    }
  }
  for (int e = 0; e < num_experts; ++e) {
    int c = tokens_per_expert[e];
    recv_tokens_per_expert[e] = (c + expert_alignment - 1) / expert_alignment * expert_alignment;
  }
  return 0;
}

/* The record for (t, r) at send_head[t, r]: header (t, r, number of the
 * token's pairs on rank r, 0); the id row with local ids (e - r*E/R) for
 * experts on rank r and -1 elsewhere; the weight row with 0 elsewhere;
 * payload and scales exactly as oracle_dispatch builds them. */
int oracle_dispatch_ranks(const int32_t* topk_idx, const float* topk_weights, const void* hidden,
                          const void* scales, int num_tokens, int topk, int num_experts,
                          int num_ranks, int hidden_size, int in_kind, int out_kind,
                          int raw_payload_bytes, int raw_scale_bytes, const int32_t* send_head,
                          uint8_t* records) {
  int32_t lay[7];
  if (num_ranks < 1 || num_experts % num_ranks || topk > 32) return -1;
  if (oracle_record_layout(topk, hidden_size, in_kind, out_kind, raw_payload_bytes,
                           raw_scale_bytes, lay) != 0)
    return -1;
  const int S = lay[0], off_ids = lay[1], off_w = lay[2], off_p = lay[3];
  const int per_rank = num_experts / num_ranks;
  /* payload and scales of one token: the same bytes oracle_dispatch writes,
   * taken from a one-pair dispatch of that token into a scratch record */
  uint8_t* one = (uint8_t*)malloc((size_t)S);
  if (!one) return -2;
  for (int t = 0; t < num_tokens; ++t) {
    int32_t zero_slot = 0;
    const void* h = NULL;
    const void* sc = NULL;
    if (in_kind == ORACLE_RAW) {
      h = (const uint8_t*)hidden + (size_t)t * raw_payload_bytes;
      sc = raw_scale_bytes ? (const void*)((const uint8_t*)scales + (size_t)t * raw_scale_bytes) : NULL;
    } else {
      h = (const uint16_t*)hidden + (size_t)t * hidden_size;
    }
    int32_t row_idx[32];
    float row_w[32];
    for (int j = 0; j < topk; ++j) {
      row_idx[j] = topk_idx[(long)t * topk + j];
      row_w[j] = topk_weights[(long)t * topk + j];
    }
    int32_t one_idx[32];
    float one_w[32];
    for (int j = 0; j < topk; ++j) {
      one_idx[j] = j == 0 ? 0 : -1;
      one_w[j] = 0.0f;
    }
    int32_t one_slots[32];
    for (int j = 0; j < topk; ++j) one_slots[j] = j == 0 ? zero_slot : -1;
    if (oracle_dispatch(one_idx, one_w, h, sc, 1, topk, hidden_size, in_kind, out_kind,
                        raw_payload_bytes, raw_scale_bytes, one_slots, one) != 0) {
      free(one);
      return -1;
    }
    for (int r = 0; r < num_ranks; ++r) {
      int s = send_head[(long)t * num_ranks + r];
      if (s < 0) continue;
      uint8_t* rec = records + (size_t)s * S;
      memset(rec, 0, (size_t)off_p);
      int nlocal = 0;
      for (int j = 0; j < topk; ++j) {
        int e = row_idx[j];
        int local = (e >= r * per_rank && e < (r + 1) * per_rank);
        int32_t id = local ? e - r * per_rank : -1;
        float w = local ? row_w[j] : 0.0f;
        nlocal += local;
        memcpy(rec + off_ids + 4 * j, &id, 4);
        memcpy(rec + off_w + 4 * j, &w, 4);
      }
      int32_t hdr[4] = {t, r, nlocal, 0};
      memcpy(rec, hdr, 16);
      memcpy(rec + off_p, one + off_p, (size_t)(S - off_p));
    }
  }
  free(one);
  return 0;
}

/* [EP] Buffer::intranode_combine: out[t] = bf16(sum over ranks r ascending
 * with send_head[t, r] >= 0 of recv_out[send_head[t, r]]), fp32 from +0. */
int oracle_combine_gather_ranks(const uint16_t* recv_out, const int32_t* send_head,
                                int num_tokens, int num_ranks, int hidden_size, uint16_t* out) {
  for (int t = 0; t < num_tokens; ++t) {
    for (int h = 0; h < hidden_size; ++h) {
      float acc = 0.0f;
      for (int r = 0; r < num_ranks; ++r) {
        int s = send_head[(long)t * num_ranks + r];
        if (s >= 0) acc = acc + oracle_bf16_to_f32(recv_out[(size_t)s * hidden_size + h]);
      }
      out[(size_t)t * hidden_size + h] = oracle_f32_to_bf16(acc);
    }
  }
  return 0;
}

/* ======================================================================== */
/* Fixed-capacity, expert-major receive buffers                              */
/* ======================================================================== */

/* [EP] Buffer::low_latency_dispatch: every expert has capacity = R * max
 * positions. Reading: expert e's pairs fill positions 0, 1, ... in ascending
 * (t, j) order (source rank s owns tokens [s*T, (s+1)*T), T = N / R, so this
 * is source-rank order); a pair past the capacity gets no position (-1).
 * src_info is the token's index within its source rank; layout_range[e, s] is
 * begin << 32 | count of e's positions taken by source rank s. */
int oracle_ll_layout(const int32_t* topk_idx, int num_tokens, int topk, int num_experts,
                     int num_ranks, int max_tokens_per_rank, int32_t* ll_slot_of,
                     int32_t* src_info, int64_t* layout_range, int32_t* recv_count) {
  if (num_ranks < 1 || num_tokens % num_ranks || max_tokens_per_rank < 1) return -1;
  const int T = num_tokens / num_ranks;
  if (T > max_tokens_per_rank) return -1;
  const long cap = (long)num_ranks * max_tokens_per_rank;
  for (long i = 0; i < (long)num_experts * cap; ++i) src_info[i] = -1;
  for (long p = 0; p < (long)num_tokens * topk; ++p) ll_slot_of[p] = -1;
  for (int e = 0; e < num_experts; ++e) {
    long pos = 0;
    for (int s = 0; s < num_ranks; ++s) {
      long begin = pos;
      for (int t = s * T; t < (s + 1) * T; ++t) {
        for (int j = 0; j < topk; ++j) {
          if (topk_idx[(long)t * topk + j] != e) continue;
          if (pos < cap) {
            ll_slot_of[(long)t * topk + j] = (int32_t)((long)e * cap + pos);
            src_info[(long)e * cap + pos] = t - s * T;
          }
          ++pos;
        }
      }
      long b = begin < cap ? begin : cap;
      long en = pos < cap ? pos : cap;
      layout_range[(long)e * num_ranks + s] = ((int64_t)b << 32) | (int64_t)(en - b);
    }
    recv_count[e] = (int32_t)(pos < cap ? pos : cap);
  }
  return 0;
}

/* The payload and scales of each token (as oracle_dispatch builds them) to
 * rows ll_slot_of[t, j] of x_out and scales_out; scale rows are scale_bytes
 * rounded up to 16 bytes apart, the pad left zero (the caller zeroes
 * scales_out). */
int oracle_dispatch_ll(const void* hidden, const void* scales, int num_tokens, int topk,
                       int hidden_size, int in_kind, int out_kind, int raw_payload_bytes,
                       int raw_scale_bytes, const int32_t* ll_slot_of, int64_t rows,
                       uint8_t* x_out, uint8_t* scales_out) {
  int32_t lay[7];
  if (topk > 32 || oracle_record_layout(topk, hidden_size, in_kind, out_kind, raw_payload_bytes,
                                        raw_scale_bytes, lay) != 0)
    return -1;
  const int S = lay[0], off_p = lay[3], off_s = lay[4], pb = lay[5], sb = lay[6];
  uint8_t* one = (uint8_t*)malloc((size_t)S);
  if (!one) return -2;
  for (int t = 0; t < num_tokens; ++t) {
    const void* h = NULL;
    const void* sc = NULL;
    if (in_kind == ORACLE_RAW) {
      h = (const uint8_t*)hidden + (size_t)t * raw_payload_bytes;
      sc = raw_scale_bytes ? (const void*)((const uint8_t*)scales + (size_t)t * raw_scale_bytes) : NULL;
    } else {
      h = (const uint16_t*)hidden + (size_t)t * hidden_size;
    }
    int32_t one_idx[32], one_slots[32];
    float one_w[32];
    for (int j = 0; j < topk; ++j) {
      one_idx[j] = j == 0 ? 0 : -1;
      one_w[j] = 0.0f;
      one_slots[j] = j == 0 ? 0 : -1;
    }
    if (oracle_dispatch(one_idx, one_w, h, sc, 1, topk, hidden_size, in_kind, out_kind,
                        raw_payload_bytes, raw_scale_bytes, one_slots, one) != 0) {
      free(one);
      return -1;
    }
    for (int j = 0; j < topk; ++j) {
      int pos = ll_slot_of[(long)t * topk + j];
      if (pos < 0 || pos >= rows) continue;
      memcpy(x_out + (size_t)pos * pb, one + off_p, (size_t)pb);
      if (sb) memcpy(scales_out + (size_t)pos * pad16(sb), one + off_s, (size_t)sb);
    }
  }
  free(one);
  return 0;
}

/* ======================================================================== */
/* Backward                                                                  */
/* ======================================================================== */

/* Backward of out[t] = sum_j w[t,j] * y[slot_of[t,j]] with respect to y and w
 * (the derivative of a weighted sum):
 *   grad_y[slot_of[t,j], h] = bf16( fp32 product w[t,j] * g[t,h] )
 *   grad_w[t,j] = fp32( sum over h of g[t,h] * y[slot_of[t,j], h] )
 * The dot product is summed in fp64, where every BF16 x BF16 product is
 * exact, and rounded to fp32 once; it bounds the fp32 sums a kernel may take
 * in any order. A pair with no slot (or one outside [0, rows)) gets
 * grad_w = 0 and writes no row; rows no pair names are left as they are.
 * y may be NULL: then grad_w is not written. */
int oracle_combine_backward(const uint16_t* grad_out, const float* topk_weights,
                            const int32_t* slot_of, const uint16_t* y, int64_t rows,
                            int num_tokens, int topk, int hidden_size, uint16_t* grad_y,
                            float* grad_w) {
  for (int t = 0; t < num_tokens; ++t) {
    const uint16_t* g = grad_out + (size_t)t * hidden_size;
    for (int j = 0; j < topk; ++j) {
      long p = (long)t * topk + j;
      int s = slot_of[p];
      int valid = s >= 0 && s < rows;
      if (valid) {
        float w = topk_weights[p];
        uint16_t* dst = grad_y + (size_t)s * hidden_size;
        for (int h = 0; h < hidden_size; ++h) {
          float prod = w * oracle_bf16_to_f32(g[h]);
          dst[h] = oracle_f32_to_bf16(prod);
        }
      }
      if (y) {
        double d = 0.0;
        if (valid) {
          const uint16_t* row = y + (size_t)s * hidden_size;
          for (int h = 0; h < hidden_size; ++h)
            d += (double)oracle_bf16_to_f32(g[h]) * (double)oracle_bf16_to_f32(row[h]);
        }
        grad_w[p] = (float)d;
      }
    }
  }
  return 0;
}

/* Backward of dispatch with respect to the token rows: each of a token's
 * pairs carried a copy of its row, so the row's gradient is the sum of the
 * copies' gradients, summed in fp32 in ascending j from +0 and rounded to
 * BF16 once (the order and precision of the combine). Payload formats are
 * taken as identity (straight-through). */
int oracle_dispatch_backward(const uint16_t* grad_in, const int32_t* slot_of, int num_tokens,
                             int topk, int hidden_size, uint16_t* grad_hidden) {
  for (int t = 0; t < num_tokens; ++t) {
    for (int h = 0; h < hidden_size; ++h) {
      float acc = 0.0f;
      for (int j = 0; j < topk; ++j) {
        int s = slot_of[(long)t * topk + j];
        if (s < 0) continue;
        acc = acc + oracle_bf16_to_f32(grad_in[(size_t)s * hidden_size + h]);
      }
      grad_hidden[(size_t)t * hidden_size + h] = oracle_f32_to_bf16(acc);
    }
  }
  return 0;
}

/* Backward of the rank-row gather out[t] = sum_r recv[send_head[t, r]]: every
 * row the sum read receives the token's gradient unchanged. */
int oracle_gather_ranks_backward(const uint16_t* grad_out, const int32_t* send_head,
                                 int num_tokens, int num_ranks, int hidden_size, int64_t rows,
                                 uint16_t* grad_recv) {
  for (int t = 0; t < num_tokens; ++t) {
    for (int r = 0; r < num_ranks; ++r) {
      int s = send_head[(long)t * num_ranks + r];
      if (s < 0 || s >= rows) continue;
      memcpy(grad_recv + (size_t)s * hidden_size, grad_out + (size_t)t * hidden_size,
             (size_t)hidden_size * 2);
    }
  }
  return 0;
}
