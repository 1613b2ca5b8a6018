/*
 * ep_c_step.c -- one whole step through libep's C ABI from plain C: no Python,
 * no PyTorch, buffers from cudaMalloc, the legacy default stream.
 *
 * usage: ep_c_step E K H A T dir
 *   dir holds the inputs as raw little-endian arrays: idx.bin (int64 [T,K]),
 *   w.bin (float32 [T,K]), tok.bin and gres.bin (bf16 bits [T,H]), eo.bin and
 *   grecv.bin (bf16 bits [rows,H]), grecv_w.bin (float32 [rows]); rows is
 *   taken from the file size.  The outputs go to dir as out_*.bin, and one
 *   line "R P npad status" to stdout.  Receive-side buffers start filled with
 *   a sentinel (0x7FC1 for payload rows, -3.0f for weights) so that the caller
 *   can check which rows the step wrote.
 *
 * Test program of the C ABI (tests/test_c_api_gpu.py builds and runs it).
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "ep.h"

static void* read_file(const char* dir, const char* name, size_t* bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE* f = fopen(path, "rb");
  if (!f) { fprintf(stderr, "cannot open %s\n", path); exit(2); }
  fseek(f, 0, SEEK_END);
  long n = ftell(f);
  fseek(f, 0, SEEK_SET);
  void* p = malloc(n > 0 ? (size_t)n : 1);
  if (n > 0 && fread(p, 1, (size_t)n, f) != (size_t)n) { fprintf(stderr, "short read %s\n", path); exit(2); }
  fclose(f);
  *bytes = (size_t)n;
  return p;
}

static void write_file(const char* dir, const char* name, const void* p, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE* f = fopen(path, "wb");
  if (!f || (bytes > 0 && fwrite(p, 1, bytes, f) != bytes)) { fprintf(stderr, "cannot write %s\n", path); exit(2); }
  fclose(f);
}

#define CK(x) do { cudaError_t e_ = (x); if (e_ != cudaSuccess) { \
  fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_)); exit(3); } } while (0)
#define EP(x) do { ep_status_t s_ = (x); if (s_ != EP_OK) { \
  fprintf(stderr, "%s: %d %s\n", #x, (int)s_, ep_last_error()); exit(4); } } while (0)

static void* dev_copy(const void* host, size_t bytes) {
  void* d = NULL;
  CK(cudaMalloc(&d, bytes > 0 ? bytes : 16));
  if (bytes > 0) CK(cudaMemcpy(d, host, bytes, cudaMemcpyHostToDevice));
  return d;
}

/* A device buffer of n 16-bit (or 32-bit) elements, each set to `pattern`. */
static void* dev_fill16(size_t n, uint16_t pattern) {
  uint16_t* h = (uint16_t*)malloc(n * 2 + 2);
  for (size_t i = 0; i < n; ++i) h[i] = pattern;
  void* d = dev_copy(h, n * 2);
  free(h);
  return d;
}
static void* dev_fill32f(size_t n, float value) {
  float* h = (float*)malloc(n * 4 + 4);
  for (size_t i = 0; i < n; ++i) h[i] = value;
  void* d = dev_copy(h, n * 4);
  free(h);
  return d;
}

static void* host_of(const void* d, size_t bytes) {
  void* h = malloc(bytes > 0 ? bytes : 1);
  if (bytes > 0) CK(cudaMemcpy(h, d, bytes, cudaMemcpyDeviceToHost));
  return h;
}

int main(int argc, char** argv) {
  if (argc != 7) { fprintf(stderr, "usage: ep_c_step E K H A T dir\n"); return 1; }
  const int64_t E = atoll(argv[1]), K = atoll(argv[2]), H = atoll(argv[3]), A = atoll(argv[4]);
  const int64_t T = atoll(argv[5]);
  const char* dir = argv[6];
  if (ep_abi_version() != EP_ABI_VERSION) { fprintf(stderr, "ABI version mismatch\n"); return 5; }

  ep_layer_config_t cfg;
  memset(&cfg, 0, sizeof cfg);
  cfg.num_experts = E;
  cfg.top_k = K;
  cfg.hidden = H;
  cfg.max_tokens = T > 0 ? T : 1;
  cfg.max_alignment = A;
  cfg.recv_capacity = 0;
  cfg.dtype = EP_DTYPE_BF16;
  uint64_t id = 0;
  size_t mem_size = 0;
  EP(ep_register_layer(cfg, &id, &mem_size));
  int64_t R = 0;
  EP(ep_recv_capacity(id, &R));

  size_t b_idx, b_w, b_tok, b_eo, b_gres, b_grecv, b_grecv_w;
  void* h_idx = read_file(dir, "idx.bin", &b_idx);
  void* h_w = read_file(dir, "w.bin", &b_w);
  void* h_tok = read_file(dir, "tok.bin", &b_tok);
  void* h_eo = read_file(dir, "eo.bin", &b_eo);
  void* h_gres = read_file(dir, "gres.bin", &b_gres);
  void* h_grecv = read_file(dir, "grecv.bin", &b_grecv);
  void* h_grecv_w = read_file(dir, "grecv_w.bin", &b_grecv_w);
  const size_t row = (size_t)H * 2;
  size_t rows = b_eo / row;
  if (rows > (size_t)R) rows = (size_t)R;

  void* hmem = NULL;
  CK(cudaMalloc(&hmem, mem_size));
  CK(cudaMemset(hmem, 0, mem_size));  /* fresh handle memory: zero-filled */
  ep_handle_t h;
  h.id = id;
  h.mem = hmem;

  void* d_idx = dev_copy(h_idx, b_idx);
  void* d_w = dev_copy(h_w, b_w);
  void* d_tok = dev_copy(h_tok, b_tok);
  void* d_gres = dev_copy(h_gres, b_gres);
  void* d_eo = dev_fill16((size_t)R * H, 0x7FC1);
  void* d_grecv = dev_fill16((size_t)R * H, 0x7FC1);
  void* d_grecv_w = dev_fill32f((size_t)R, -1.0f);
  CK(cudaMemcpy(d_eo, h_eo, rows * row, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(d_grecv, h_grecv, rows * row, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(d_grecv_w, h_grecv_w, rows * 4, cudaMemcpyHostToDevice));
  void* d_counts = dev_fill32f((size_t)E, 0.0f);
  void* d_offsets = dev_fill32f((size_t)E + 1, 0.0f);
  void* d_slots = dev_fill32f((size_t)(T * K), 0.0f);
  void* d_recv = dev_fill16((size_t)R * H, 0x7FC1);
  void* d_recv_w = dev_fill32f((size_t)R, -3.0f);
  void* d_res = dev_fill16((size_t)T * H, 0x7FC1);
  void* d_gexp = dev_fill16((size_t)R * H, 0x7FC1);
  void* d_gtok = dev_fill16((size_t)T * H, 0x7FC1);
  void* d_gtw = dev_fill32f((size_t)(T * K), -3.0f);

  EP(ep_prepare(h, (const int64_t*)d_idx, T, (int32_t*)d_counts, A, NULL));
  EP(ep_dispatch(h, (const int64_t*)d_idx, T, d_tok, (const float*)d_w, d_recv, (float*)d_recv_w, NULL));
  EP(ep_combine(h, d_eo, T, d_res, NULL));
  EP(ep_combine_bwd(h, d_gres, T, d_gexp, NULL));
  EP(ep_dispatch_bwd(h, d_grecv, (const float*)d_grecv_w, T, d_gtok, (float*)d_gtw, NULL));
  EP(ep_expert_offsets(h, (int32_t*)d_offsets, NULL));
  EP(ep_token_slots(h, (int32_t*)d_slots, T, NULL));
  ep_info_t info;
  EP(ep_read_info(h, &info, NULL));
  CK(cudaDeviceSynchronize());

  struct { const char* name; void* d; size_t bytes; } outs[] = {
      {"out_counts.bin", d_counts, (size_t)E * 4},
      {"out_offsets.bin", d_offsets, (size_t)(E + 1) * 4},
      {"out_slots.bin", d_slots, (size_t)(T * K) * 4},
      {"out_recv.bin", d_recv, (size_t)R * row},
      {"out_recv_w.bin", d_recv_w, (size_t)R * 4},
      {"out_result.bin", d_res, (size_t)T * row},
      {"out_gexp.bin", d_gexp, (size_t)R * row},
      {"out_gtok.bin", d_gtok, (size_t)T * row},
      {"out_gtw.bin", d_gtw, (size_t)(T * K) * 4},
  };
  for (size_t i = 0; i < sizeof outs / sizeof outs[0]; ++i) {
    void* hbuf = host_of(outs[i].d, outs[i].bytes);
    write_file(dir, outs[i].name, hbuf, outs[i].bytes);
    free(hbuf);
  }
  printf("%lld %d %d %u\n", (long long)R, info.used_rows, info.padding_rows, info.status);
  return 0;
}
