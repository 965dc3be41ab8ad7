/* A plain C11 caller of the device path: reads one workload's inputs from
 * files, allocates device memory with the CUDA runtime, runs moe_layout,
 * moe_dispatch (BF16 rows to FP8 records) and moe_combine (grouped by rank)
 * through libmoe.so on the default stream, then moe_layout_dispatch on the
 * first 128 tokens (layout and dispatch in one kernel), then the
 * fixed-capacity path (moe_layout_ll_dispatch) on the first R * 16 tokens,
 * and writes slot_of, the records, the combined rows and the fixed-capacity
 * outputs back to files for the test that builds and runs it
 * (tests/test_gpu_c_consumer.py) to check against the oracle.
 *   device_path DIR   with DIR/meta.txt = "N k E R H P" and ids.bin, w.bin,
 *   x.bin (bf16 bits), y.bin (bf16 bits, P rows) */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "moe.h"

static int fail(const char* what, int code) {
  fprintf(stderr, "%s failed: %d (%s)\n", what, code, code < 0 ? moe_strerror(code) : "cuda");
  return 1;
}

static void* read_file(const char* dir, const char* name, size_t bytes) {
  char path[1024];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE* f = fopen(path, "rb");
  if (!f) return NULL;
  void* p = malloc(bytes ? bytes : 1);
  size_t got = fread(p, 1, bytes, f);
  fclose(f);
  if (got != bytes) {
    free(p);
    return NULL;
  }
  return p;
}

static int write_file(const char* dir, const char* name, const void* p, size_t bytes) {
  char path[1024];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE* f = fopen(path, "wb");
  if (!f) return 1;
  size_t put = fwrite(p, 1, bytes, f);
  fclose(f);
  return put != bytes;
}

#define CUDA(x)                                  \
  do {                                           \
    cudaError_t e_ = (x);                        \
    if (e_ != cudaSuccess) return fail(#x, (int)e_); \
  } while (0)

int main(int argc, char** argv) {
  if (argc != 2) return fail("usage: device_path DIR", -1);
  const char* dir = argv[1];
  char path[1024];
  snprintf(path, sizeof path, "%s/meta.txt", dir);
  FILE* m = fopen(path, "r");
  if (!m) return fail("meta.txt", -1);
  int n, k, e, r, h, p;
  if (fscanf(m, "%d %d %d %d %d %d", &n, &k, &e, &r, &h, &p) != 6) return fail("meta.txt", -1);
  fclose(m);

  const size_t pairs = (size_t)n * k;
  int32_t* ids = read_file(dir, "ids.bin", pairs * 4);
  float* w = read_file(dir, "w.bin", pairs * 4);
  uint16_t* x = read_file(dir, "x.bin", (size_t)n * h * 2);
  uint16_t* y = read_file(dir, "y.bin", (size_t)p * h * 2);
  if (!ids || !w || !x || !y) return fail("input files", -1);

  moe_desc_t d;
  memset(&d, 0, sizeof d);
  d.num_tokens = n;
  d.topk = k;
  d.num_experts = e;
  d.num_ranks = r;
  d.hidden = h;
  d.in_kind = MOE_PAYLOAD_BF16;
  d.out_kind = MOE_PAYLOAD_FP8_E4M3_B128;
  moe_record_layout_t lay;
  int rc = moe_record_layout(&d, &lay);
  if (rc) return fail("moe_record_layout", rc);
  const size_t ws_bytes = moe_workspace_size(&d);
  const size_t rec_bytes = pairs * (size_t)lay.record_bytes;

  int32_t *d_ids, *d_tpe, *d_tpr, *d_eo, *d_ro, *d_slot, *d_slot2, *d_src;
  uint8_t *d_mask, *d_rec, *d_rec2;
  float* d_w;
  void *d_x, *d_y, *d_out, *d_ws;
  CUDA(cudaMalloc((void**)&d_ids, pairs * 4));
  CUDA(cudaMalloc((void**)&d_w, pairs * 4));
  CUDA(cudaMalloc(&d_x, (size_t)n * h * 2));
  CUDA(cudaMalloc(&d_y, (size_t)(p ? p : 1) * h * 2));
  CUDA(cudaMalloc(&d_out, (size_t)n * h * 2));
  CUDA(cudaMalloc((void**)&d_tpe, (size_t)e * 4));
  CUDA(cudaMalloc((void**)&d_tpr, (size_t)r * 4));
  CUDA(cudaMalloc((void**)&d_mask, (size_t)n * r));
  CUDA(cudaMalloc((void**)&d_eo, (size_t)(e + 1) * 4));
  CUDA(cudaMalloc((void**)&d_ro, (size_t)(r + 1) * 4));
  CUDA(cudaMalloc((void**)&d_slot, pairs * 4));
  CUDA(cudaMalloc((void**)&d_slot2, pairs * 4));
  CUDA(cudaMalloc((void**)&d_src, pairs * 4));
  CUDA(cudaMalloc((void**)&d_rec, rec_bytes));
  CUDA(cudaMalloc((void**)&d_rec2, rec_bytes));
  CUDA(cudaMalloc(&d_ws, ws_bytes));
  CUDA(cudaMemcpy(d_ids, ids, pairs * 4, cudaMemcpyHostToDevice));
  CUDA(cudaMemcpy(d_w, w, pairs * 4, cudaMemcpyHostToDevice));
  CUDA(cudaMemcpy(d_x, x, (size_t)n * h * 2, cudaMemcpyHostToDevice));
  CUDA(cudaMemcpy(d_y, y, (size_t)p * h * 2, cudaMemcpyHostToDevice));

  rc = moe_layout(&d, d_ids, d_tpe, d_tpr, d_mask, d_eo, d_ro, d_slot, d_src, d_ws, ws_bytes, NULL);
  if (rc) return fail("moe_layout", rc);
  int32_t status = -100;
  rc = moe_layout_status(d_ws, &status, NULL);
  if (rc || status) return fail("moe_layout_status", rc ? rc : status);
  rc = moe_dispatch(&d, d_ids, d_w, d_x, NULL, d_slot, d_rec, rec_bytes, NULL);
  if (rc) return fail("moe_dispatch", rc);
  moe_desc_t dc = d;
  dc.in_kind = MOE_PAYLOAD_BF16;
  dc.out_kind = MOE_PAYLOAD_BF16;
  rc = moe_combine(&dc, MOE_COMBINE_TOPK_RANKS, d_y, (int64_t)p, d_ids, d_w, d_slot, d_out, NULL);
  if (rc) return fail("moe_combine", rc);
  CUDA(cudaDeviceSynchronize());

  int32_t* slot = malloc(pairs * 4);
  uint8_t* rec = malloc((size_t)p * lay.record_bytes + 1);
  uint16_t* out = malloc((size_t)n * h * 2);
  CUDA(cudaMemcpy(slot, d_slot, pairs * 4, cudaMemcpyDeviceToHost));
  CUDA(cudaMemcpy(rec, d_rec, (size_t)p * lay.record_bytes, cudaMemcpyDeviceToHost));
  CUDA(cudaMemcpy(out, d_out, (size_t)n * h * 2, cudaMemcpyDeviceToHost));
  if (write_file(dir, "slot_of.bin", slot, pairs * 4) ||
      write_file(dir, "records.bin", rec, (size_t)p * lay.record_bytes) ||
      write_file(dir, "out.bin", out, (size_t)n * h * 2))
    return fail("output files", -1);

  /* The one-call form on the first n_small tokens: at most 2048 pairs, so
     layout and dispatch run as one kernel. */
  const int n_small = n < 128 ? n : 128;
  moe_desc_t ds = d;
  ds.num_tokens = n_small;
  const size_t small_pairs = (size_t)n_small * k;
  const size_t small_rec = (small_pairs < (size_t)p ? small_pairs : (size_t)p) * lay.record_bytes;
  rc = moe_layout_dispatch(&ds, d_ids, d_w, d_x, NULL, d_tpe, d_tpr, d_mask, d_eo, d_ro, d_slot2, d_src, d_ws,
                           ws_bytes, d_rec2, rec_bytes, NULL);
  if (rc) return fail("moe_layout_dispatch", rc);
  status = -100;
  rc = moe_layout_status(d_ws, &status, NULL);
  if (rc || status) return fail("moe_layout_status (one call)", rc ? rc : status);
  CUDA(cudaMemcpy(slot, d_slot2, small_pairs * 4, cudaMemcpyDeviceToHost));
  CUDA(cudaMemcpy(rec, d_rec2, small_rec, cudaMemcpyDeviceToHost));
  if (write_file(dir, "slot_of_small.bin", slot, small_pairs * 4) ||
      write_file(dir, "records_small.bin", rec, small_rec))
    return fail("output files", -1);
  /* The fixed-capacity path on the first R * T tokens: positions
     [E * R * T] rows, then the payload and scales of every pair gathered in
     pair order (zero rows for pairs past the capacity or without an expert). */
  const int T = 16;
  const int n_ll = r * T <= n ? r * T : n - n % r;
  moe_desc_t dl = d;
  dl.num_tokens = n_ll;
  const size_t ll_pairs = (size_t)n_ll * k;
  const size_t cap = (size_t)r * T, rows_ll = (size_t)e * cap;
  const size_t pb = (size_t)lay.payload_bytes, sb = ((size_t)lay.scale_bytes + 15) & ~(size_t)15;
  int32_t *d_llslot, *d_info, *d_cnt;
  int64_t* d_range;
  uint8_t *d_xo, *d_so;
  CUDA(cudaMalloc((void**)&d_llslot, ll_pairs * 4));
  CUDA(cudaMalloc((void**)&d_info, rows_ll * 4));
  CUDA(cudaMalloc((void**)&d_range, (size_t)e * r * 8));
  CUDA(cudaMalloc((void**)&d_cnt, (size_t)e * 4));
  CUDA(cudaMalloc((void**)&d_xo, rows_ll * pb));
  CUDA(cudaMalloc((void**)&d_so, rows_ll * sb));
  rc = moe_layout_ll_dispatch(&dl, d_ids, d_x, NULL, d_tpe, d_tpr, d_mask, d_eo, d_ro, d_slot2, d_src, T, d_llslot,
                              d_info, d_range, d_cnt, d_ws, ws_bytes, d_xo, rows_ll * pb, d_so, rows_ll * sb, NULL);
  if (rc) return fail("moe_layout_ll_dispatch", rc);
  status = -100;
  rc = moe_layout_status(d_ws, &status, NULL);
  if (rc || status) return fail("moe_layout_status (fixed capacity)", rc ? rc : status);
  int32_t* llslot = malloc(ll_pairs * 4);
  int32_t* info = malloc(rows_ll * 4);
  int64_t* range = malloc((size_t)e * r * 8);
  int32_t* cnt = malloc((size_t)e * 4);
  uint8_t* xg = calloc(ll_pairs, pb);
  uint8_t* sg = calloc(ll_pairs, sb);
  if (!llslot || !info || !range || !cnt || !xg || !sg) return fail("host memory", -1);
  CUDA(cudaMemcpy(llslot, d_llslot, ll_pairs * 4, cudaMemcpyDeviceToHost));
  CUDA(cudaMemcpy(info, d_info, rows_ll * 4, cudaMemcpyDeviceToHost));
  CUDA(cudaMemcpy(range, d_range, (size_t)e * r * 8, cudaMemcpyDeviceToHost));
  CUDA(cudaMemcpy(cnt, d_cnt, (size_t)e * 4, cudaMemcpyDeviceToHost));
  for (size_t q = 0; q < ll_pairs; ++q) {
    const int32_t pos = llslot[q];
    if (pos < 0 || (size_t)pos >= rows_ll) continue;
    CUDA(cudaMemcpy(xg + q * pb, d_xo + (size_t)pos * pb, pb, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(sg + q * sb, d_so + (size_t)pos * sb, sb, cudaMemcpyDeviceToHost));
  }
  if (write_file(dir, "ll_slot_of.bin", llslot, ll_pairs * 4) ||
      write_file(dir, "ll_src_info.bin", info, rows_ll * 4) ||
      write_file(dir, "ll_layout_range.bin", range, (size_t)e * r * 8) ||
      write_file(dir, "ll_recv_count.bin", cnt, (size_t)e * 4) ||
      write_file(dir, "ll_x_pairs.bin", xg, ll_pairs * pb) || write_file(dir, "ll_s_pairs.bin", sg, ll_pairs * sb))
    return fail("output files", -1);
  printf("ok records=%d record_bytes=%d ll_tokens=%d\n", p, (int)lay.record_bytes, n_ll);
  return 0;
}
