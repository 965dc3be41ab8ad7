/* A plain C11 caller of libmoe.so's host-only entry points: the record layout
 * of a descriptor, the layout workspace size, status names, argument errors,
 * and one record packed and unpacked. Prints key=value lines for the test
 * that builds and runs it (tests/test_c_consumer.py). */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "moe.h"

static moe_desc_t desc(int32_t n, int32_t k, int32_t e, int32_t r, int32_t h, int32_t in_kind,
                       int32_t out_kind) {
  moe_desc_t d;
  memset(&d, 0, sizeof d);
  d.num_tokens = n;
  d.topk = k;
  d.num_experts = e;
  d.num_ranks = r;
  d.hidden = h;
  d.in_kind = in_kind;
  d.out_kind = out_kind;
  return d;
}

int main(void) {
  /* record layout of the prefill workload's FP8 records */
  moe_desc_t d = desc(4096, 8, 256, 8, 7168, MOE_PAYLOAD_BF16, MOE_PAYLOAD_FP8_E4M3_B128);
  moe_record_layout_t lay;
  int rc = moe_record_layout(&d, &lay);
  printf("fp8_rc=%d\n", rc);
  printf("fp8_record_bytes=%d\n", (int)lay.record_bytes);
  printf("fp8_off_ids=%d\nfp8_off_weights=%d\nfp8_off_payload=%d\nfp8_off_scales=%d\n",
         (int)lay.off_ids, (int)lay.off_weights, (int)lay.off_payload, (int)lay.off_scales);
  printf("fp8_payload_bytes=%d\nfp8_scale_bytes=%d\n", (int)lay.payload_bytes, (int)lay.scale_bytes);
  printf("workspace_bytes=%zu\n", moe_workspace_size(&d));

  /* argument errors come back as codes, with names */
  moe_desc_t bad = desc(16, 2, 15, 2, 1024, MOE_PAYLOAD_BF16, MOE_PAYLOAD_BF16);  /* E % R != 0 */
  rc = moe_record_layout(&bad, &lay);
  printf("bad_ranks_rc=%d\n", rc);
  printf("bad_ranks_name=%s\n", moe_strerror(rc));
  rc = moe_record_layout(NULL, &lay);
  printf("null_desc_rc=%d\n", rc);

  /* one BF16 record packed and unpacked on the host */
  moe_desc_t small = desc(4, 2, 16, 2, 64, MOE_PAYLOAD_BF16, MOE_PAYLOAD_BF16);
  rc = moe_record_layout(&small, &lay);
  printf("bf16_rc=%d\nbf16_record_bytes=%d\n", rc, (int)lay.record_bytes);
  int32_t ids[2] = {5, 11};
  float w[2] = {0.75f, 0.25f};
  uint16_t row[64];
  for (int i = 0; i < 64; ++i) row[i] = (uint16_t)(0x3F80 + i);
  uint8_t rec[4096];
  memset(rec, 0xAB, sizeof rec);
  rc = moe_pack_record(&small, 3, 1, 11, ids, w, row, NULL, rec);
  printf("pack_rc=%d\n", rc);
  int32_t t = -1, j = -1, e = -1, ids2[2] = {0, 0};
  float w2[2] = {0, 0};
  uint16_t row2[64];
  rc = moe_unpack_record(&small, rec, &t, &j, &e, ids2, w2, row2, NULL);
  printf("unpack_rc=%d\nsrc_token=%d\nslot_j=%d\nexpert=%d\n", rc, (int)t, (int)j, (int)e);
  printf("ids_equal=%d\nweights_equal=%d\nrow_equal=%d\n", ids2[0] == 5 && ids2[1] == 11,
         w2[0] == 0.75f && w2[1] == 0.25f, memcmp(row, row2, sizeof row) == 0);
  return 0;
}
