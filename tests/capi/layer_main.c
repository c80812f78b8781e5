/*
 * One routed-MoE layer through the library's C ABI alone: no Python, no
 * PyTorch, only the CUDA runtime for memory and a stream.
 *
 *   layer_main DIR T H K E R I [fused]
 *
 * reads from DIR the raw little-endian arrays x.bin (BF16 [T,H]), idx.bin
 * (int64 [T,K]), w.bin (fp32 [T,K]), w13.bin (e4m3 [E,2I,H]), s13.bin (fp32
 * [E,2I/128,H/128]), w2.bin (e4m3 [E,H,I]) and s2.bin (fp32 [E,H/128,I/128]),
 * runs moe_dispatch, moe_expert_compute and moe_combine on one stream (with
 * "fused": moe_dispatch_quant, moe_gemm_gateup_down and moe_combine, the
 * layer's default path), and writes y.bin (BF16 [T,H]), counts.bin (int32
 * [E]), src_map.bin (int32 [T,K]) and status.bin (int32 [2]).  Exits non-zero
 * on any error.
 */
#include <cuda_runtime.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "moe.h"

static void die(const char* what) {
  fprintf(stderr, "layer_main: %s\n", what);
  exit(1);
}

static void check_cuda(cudaError_t e, const char* what) {
  if (e != cudaSuccess) {
    fprintf(stderr, "layer_main: %s: %s\n", what, cudaGetErrorString(e));
    exit(1);
  }
}

static void check_moe(moe_status s, const char* what) {
  if (s != MOE_OK) {
    fprintf(stderr, "layer_main: %s returned %s\n", what, moe_status_string(s));
    exit(1);
  }
}

static void* read_file(const char* dir, const char* name, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE* f = fopen(path, "rb");
  if (!f) die(path);
  void* buf = malloc(bytes ? bytes : 1);
  if (!buf) die("out of host memory");
  if (bytes && fread(buf, 1, bytes, f) != bytes) die(path);
  fclose(f);
  return buf;
}

static void write_file(const char* dir, const char* name, const void* buf, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE* f = fopen(path, "wb");
  if (!f) die(path);
  if (bytes && fwrite(buf, 1, bytes, f) != bytes) die(path);
  fclose(f);
}

/* Device copy of a host file. */
static void* upload(const char* dir, const char* name, size_t bytes) {
  void* h = read_file(dir, name, bytes);
  void* d = NULL;
  check_cuda(cudaMalloc(&d, bytes ? bytes : 16), "cudaMalloc");
  check_cuda(cudaMemcpy(d, h, bytes, cudaMemcpyHostToDevice), "cudaMemcpy to device");
  free(h);
  return d;
}

static void* dev_alloc(size_t bytes) {
  void* d = NULL;
  check_cuda(cudaMalloc(&d, bytes ? bytes : 16), "cudaMalloc");
  return d;
}

int main(int argc, char** argv) {
  if (argc != 8 && !(argc == 9 && strcmp(argv[8], "fused") == 0))
    die("usage: layer_main DIR T H K E R I [fused]");
  const int fused = argc == 9;
  const char* dir = argv[1];
  const int T = atoi(argv[2]), H = atoi(argv[3]), K = atoi(argv[4]);
  const int E = atoi(argv[5]), R = atoi(argv[6]), I = atoi(argv[7]);
  const size_t rows = (size_t)E * R;

  void* x = upload(dir, "x.bin", (size_t)T * H * 2);
  void* idx = upload(dir, "idx.bin", (size_t)T * K * 8);
  void* w = upload(dir, "w.bin", (size_t)T * K * 4);
  void* w13 = upload(dir, "w13.bin", (size_t)E * 2 * I * H);
  void* s13 = upload(dir, "s13.bin", (size_t)E * (2 * I / 128) * (H / 128) * 4);
  void* w2 = upload(dir, "w2.bin", (size_t)E * H * I);
  void* s2 = upload(dir, "s2.bin", (size_t)E * (H / 128) * (I / 128) * 4);

  void* out = dev_alloc(rows * H * 2);
  int32_t* counts = (int32_t*)dev_alloc((size_t)E * 4);
  int32_t* src_map = (int32_t*)dev_alloc((size_t)T * K * 4);
  int32_t* status = (int32_t*)dev_alloc(8);
  void* y = dev_alloc((size_t)T * H * 2);
  const size_t ws_d = moe_dispatch_workspace_size(T, K, E);
  void* wsd = dev_alloc(ws_d);

  cudaStream_t stream;
  check_cuda(cudaStreamCreate(&stream), "cudaStreamCreate");
  moe_stream_t s = (moe_stream_t)stream;
  if (fused) {
    /* FP8 activations and Z, and the fused GEMM launch's scratch, as separate
       caller-owned buffers */
    uint8_t* xq = (uint8_t*)dev_alloc(rows * H);
    float* xs = (float*)dev_alloc(rows * (H / 128) * 4);
    uint8_t* zq = (uint8_t*)dev_alloc(rows * I);
    float* zs = (float*)dev_alloc(rows * (I / 128) * 4);
    const size_t sync_bytes = moe_gemm_gateup_down_sync_size(E, R, 0);
    if (sync_bytes == 0) die("moe_gemm_gateup_down_sync_size rejected the sizes");
    void* sync = dev_alloc(sync_bytes);
    check_moe(moe_dispatch_quant(x, (const int64_t*)idx, (const float*)w, T, H, K, E, R, xq, xs,
                                 counts, src_map, status, wsd, ws_d, s),
              "moe_dispatch_quant");
    check_moe(moe_gemm_gateup_down(xq, xs, counts, E, R, 0, H, I, (const uint8_t*)w13,
                                   (const float*)s13, (const uint8_t*)w2, (const float*)s2, zq,
                                   zs, out, status, sync, sync_bytes, 0, s),
              "moe_gemm_gateup_down");
  } else {
    const size_t ws_c = moe_expert_compute_workspace_size(E, R, H, I);
    if (ws_c == 0) die("moe_expert_compute_workspace_size rejected the sizes");
    void* wsc = dev_alloc(ws_c);
    void* recv = dev_alloc(rows * H * 2);
    check_moe(moe_dispatch(x, (const int64_t*)idx, (const float*)w, T, H, K, E, R, recv, counts,
                           src_map, status, wsd, ws_d, s),
              "moe_dispatch");
    check_moe(moe_expert_compute(recv, counts, E, R, H, I, (const uint8_t*)w13, (const float*)s13,
                                 (const uint8_t*)w2, (const float*)s2, out, status, wsc, ws_c, s),
              "moe_expert_compute");
  }
  check_moe(moe_combine(out, src_map, (const float*)w, T, H, K, E, R, y, s), "moe_combine");
  check_cuda(cudaStreamSynchronize(stream), "cudaStreamSynchronize");

  void* h = malloc((size_t)T * H * 2 + (size_t)E * 4 + (size_t)T * K * 4 + 8 + 16);
  if (!h) die("out of host memory");
  check_cuda(cudaMemcpy(h, y, (size_t)T * H * 2, cudaMemcpyDeviceToHost), "copy y");
  write_file(dir, "y.bin", h, (size_t)T * H * 2);
  check_cuda(cudaMemcpy(h, counts, (size_t)E * 4, cudaMemcpyDeviceToHost), "copy counts");
  write_file(dir, "counts.bin", h, (size_t)E * 4);
  check_cuda(cudaMemcpy(h, src_map, (size_t)T * K * 4, cudaMemcpyDeviceToHost), "copy src_map");
  write_file(dir, "src_map.bin", h, (size_t)T * K * 4);
  check_cuda(cudaMemcpy(h, status, 8, cudaMemcpyDeviceToHost), "copy status");
  write_file(dir, "status.bin", h, 8);
  free(h);
  printf("layer_main: ok\n");
  return 0;
}
