/* A plain C caller of libfastocr.so that uses nothing but include/fastocr.h
 * and the CUDA runtime: no Python, no torch. It reads one layer's inputs from
 * raw files, runs the full, focal and gather calls on the current device, and
 * writes the outputs and the selection to raw files. test_abi_consumer.py
 * builds it with gcc and checks what it writes against the fp64 oracle.
 *
 * usage: abi_consumer DIR B H_q H_kv d page max_pages num_pages max_img tau
 * reads  DIR/q.bin    bf16 [B, H_q, d]
 *        DIR/k.bin    bf16 [num_pages, H_kv, page, d]   (and DIR/v.bin)
 *        DIR/bt.bin   int32 [B, max_pages]
 *        DIR/len.bin  int32 [B]
 *        DIR/img.bin  int32 [B, 2]   (start, N_img)
 * writes DIR/out_full.bin, DIR/out_focal.bin, DIR/out_sparse.bin  bf16 [B, H_q, d]
 *        DIR/idx.bin  int32 [B, stride]   DIR/kept.bin  int32 [B]
 *        DIR/stride.txt, DIR/status.txt (device status word)
 * Exit status 0 on success; any failed call prints its status text. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "fastocr.h"

static char path_buf[4096];

static const char* path_of(const char* dir, const char* name) {
  snprintf(path_buf, sizeof(path_buf), "%s/%s", dir, name);
  return path_buf;
}

static void* read_file(const char* dir, const char* name, size_t bytes) {
  FILE* f = fopen(path_of(dir, name), "rb");
  void* buf = malloc(bytes ? bytes : 1);
  if (!f || !buf || fread(buf, 1, bytes, f) != bytes) {
    fprintf(stderr, "cannot read %zu bytes of %s\n", bytes, name);
    exit(2);
  }
  fclose(f);
  return buf;
}

static void write_file(const char* dir, const char* name, const void* buf, size_t bytes) {
  FILE* f = fopen(path_of(dir, name), "wb");
  if (!f || fwrite(buf, 1, bytes, f) != bytes) {
    fprintf(stderr, "cannot write %s\n", name);
    exit(2);
  }
  fclose(f);
}

static void* to_device(const void* host, size_t bytes) {
  void* dev = NULL;
  if (cudaMalloc(&dev, bytes ? bytes : 16) != cudaSuccess ||
      cudaMemcpy(dev, host, bytes, cudaMemcpyHostToDevice) != cudaSuccess) {
    fprintf(stderr, "device copy failed\n");
    exit(3);
  }
  return dev;
}

static void* device_zeros(size_t bytes) {
  void* dev = NULL;
  if (cudaMalloc(&dev, bytes) != cudaSuccess || cudaMemset(dev, 0, bytes) != cudaSuccess) {
    fprintf(stderr, "device allocation failed\n");
    exit(3);
  }
  return dev;
}

static void check(const char* what, fastocr_status st) {
  if (st != FASTOCR_OK) {
    fprintf(stderr, "%s: %s\n", what, fastocr_status_string(st));
    exit(4);
  }
}

static void save(const char* dir, const char* name, const void* dev, size_t bytes) {
  void* host = malloc(bytes);
  if (!host || cudaMemcpy(host, dev, bytes, cudaMemcpyDeviceToHost) != cudaSuccess) {
    fprintf(stderr, "device read of %s failed\n", name);
    exit(3);
  }
  write_file(dir, name, host, bytes);
  free(host);
}

int main(int argc, char** argv) {
  if (argc != 11) {
    fprintf(stderr, "usage: %s DIR B H_q H_kv d page max_pages num_pages max_img tau\n", argv[0]);
    return 1;
  }
  const char* dir = argv[1];
  fastocr_dims dims;
  memset(&dims, 0, sizeof(dims));
  dims.batch = atoi(argv[2]);
  dims.num_q_heads = atoi(argv[3]);
  dims.num_kv_heads = atoi(argv[4]);
  dims.head_dim = atoi(argv[5]);
  dims.dtype = FASTOCR_DTYPE_BF16;
  dims.page_size = atoi(argv[6]);
  dims.max_pages_per_seq = atoi(argv[7]);
  const int num_pages = atoi(argv[8]);
  dims.max_img_tokens = atoi(argv[9]);
  dims.num_layers = 1;
  const double tau = atof(argv[10]);

  const size_t B = (size_t)dims.batch;
  const size_t q_bytes = B * dims.num_q_heads * dims.head_dim * 2;
  const size_t kv_bytes = (size_t)num_pages * dims.num_kv_heads * dims.page_size * dims.head_dim * 2;
  /* the keep capacity: ceil(tau * max_img), as the header asks of idx_stride */
  const int stride = (int)ceil(tau * dims.max_img_tokens - 1e-9);

  void* q = read_file(dir, "q.bin", q_bytes);
  void* k = read_file(dir, "k.bin", kv_bytes);
  void* v = read_file(dir, "v.bin", kv_bytes);
  void* bt = read_file(dir, "bt.bin", B * dims.max_pages_per_seq * 4);
  void* len = read_file(dir, "len.bin", B * 4);
  void* img = read_file(dir, "img.bin", B * 8);

  fastocr_handle* h = NULL;
  check("fastocr_create", fastocr_create(&dims, &h));
  fastocr_kv kv;
  kv.k = to_device(k, kv_bytes);
  kv.v = to_device(v, kv_bytes);
  kv.block_table = (const int32_t*)to_device(bt, B * dims.max_pages_per_seq * 4);
  kv.seq_len = (const int32_t*)to_device(len, B * 4);
  kv.num_pages = num_pages;
  const int32_t* d_img = (const int32_t*)to_device(img, B * 8);
  const void* d_q = to_device(q, q_bytes);
  void* out_full = device_zeros(q_bytes);
  void* out_focal = device_zeros(q_bytes);
  void* out_sparse = device_zeros(q_bytes);
  int32_t* idx = (int32_t*)device_zeros(B * stride * 4);
  int32_t* kept = (int32_t*)device_zeros(B * 4);

  /* one layer three ways, in stream order on the default stream */
  check("fastocr_full_attend", fastocr_full_attend(h, d_q, &kv, out_full, NULL));
  check("fastocr_focal_attend",
        fastocr_focal_attend(h, d_q, &kv, d_img, tau, out_focal, idx, stride, kept, -1, NULL));
  check("fastocr_sparse_attend",
        fastocr_sparse_attend(h, d_q, &kv, d_img, idx, stride, kept, out_sparse, NULL));
  int32_t status = -1;
  check("fastocr_device_status", fastocr_device_status(h, &status, NULL));

  save(dir, "out_full.bin", out_full, q_bytes);
  save(dir, "out_focal.bin", out_focal, q_bytes);
  save(dir, "out_sparse.bin", out_sparse, q_bytes);
  save(dir, "idx.bin", idx, B * stride * 4);
  save(dir, "kept.bin", kept, B * 4);
  FILE* f = fopen(path_of(dir, "stride.txt"), "w");
  if (!f) return 2;
  fprintf(f, "%d\n", stride);
  fclose(f);
  f = fopen(path_of(dir, "status.txt"), "w");
  if (!f) return 2;
  fprintf(f, "%d\n", status);
  fclose(f);

  check("fastocr_destroy", fastocr_destroy(h));
  cudaFree((void*)kv.k);
  cudaFree((void*)kv.v);
  cudaFree((void*)kv.block_table);
  cudaFree((void*)kv.seq_len);
  cudaFree((void*)d_img);
  cudaFree((void*)d_q);
  cudaFree(out_full);
  cudaFree(out_focal);
  cudaFree(out_sparse);
  cudaFree(idx);
  cudaFree(kept);
  free(q);
  free(k);
  free(v);
  free(bt);
  free(len);
  free(img);
  return 0;
}
