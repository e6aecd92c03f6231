/*
 * A plain C (C11) program that runs a chunk stream on the GPU through the
 * library's C ABI alone (include/savgb.h), with its own device buffers from
 * the CUDA runtime: no Python, no PyTorch.  The GPU test suite writes the
 * inputs, runs this program, and checks its output against the oracle and
 * against the same stream run through the Python binding.
 *
 * usage: abi_c_stream DIR B H D F GRID_H GRID_W REF_FRAMES BOUNDARY_FRAMES
 *                     REF_T CHUNKS STEPS SHIFT
 * reads  DIR/ref_k.bin, DIR/ref_v.bin (bf16 [B][ref_frames*h*w][H][D]),
 *        DIR/w_o.bin (bf16 [H*D][H*D]), DIR/x_<c>.bin (fp32 [B*N][H*D]) and
 *        DIR/{q,k,v}_<c>_<s>.bin (bf16 [B][N][H][D]) for chunk c, step s;
 * writes DIR/out_<c>.bin: x after chunk c's last step.
 * Exits 0 on success, 1 with a message on the first failed call.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime_api.h>

#include "savgb.h"

static int fail_call(const char* what, int status) {
  fprintf(stderr, "%s failed: %s (%s)\n", what, savgb_status_string(status), savgb_last_error());
  return 1;
}

static int fail_cuda(const char* what, cudaError_t e) {
  fprintf(stderr, "%s failed: %s\n", what, cudaGetErrorString(e));
  return 1;
}

/* Reads exactly `bytes` from DIR/name into a new host buffer. */
static void* read_file(const char* dir, const char* name, size_t bytes) {
  char path[4096];
  FILE* f;
  void* buf;
  snprintf(path, sizeof path, "%s/%s", dir, name);
  f = fopen(path, "rb");
  if (!f) {
    fprintf(stderr, "cannot open %s\n", path);
    return NULL;
  }
  buf = malloc(bytes ? bytes : 1);
  if (buf && fread(buf, 1, bytes, f) != bytes) {
    fprintf(stderr, "short read from %s\n", path);
    free(buf);
    buf = NULL;
  }
  fclose(f);
  return buf;
}

static int write_file(const char* dir, const char* name, const void* buf, size_t bytes) {
  char path[4096];
  FILE* f;
  size_t n;
  snprintf(path, sizeof path, "%s/%s", dir, name);
  f = fopen(path, "wb");
  if (!f) return 1;
  n = fwrite(buf, 1, bytes, f);
  fclose(f);
  return n == bytes ? 0 : 1;
}

/* Uploads DIR/name (bytes long) to the device buffer dst. */
static int upload(const char* dir, const char* name, void* dst, size_t bytes) {
  void* h = read_file(dir, name, bytes);
  cudaError_t e;
  if (!h) return 1;
  e = cudaMemcpy(dst, h, bytes, cudaMemcpyHostToDevice);
  free(h);
  return e == cudaSuccess ? 0 : fail_cuda("cudaMemcpy (upload)", e);
}

int main(int argc, char** argv) {
  chunk_stream_config_t cfg;
  chunk_stream_t* s = NULL;
  const char* dir;
  int B, H, D, F, gh, gw, ref_frames, bnd_frames, ref_t, chunks, steps, c, st, rc;
  double shift, dt[64];
  size_t n_tok, n_ref, tok_bytes, ref_bytes, x_bytes, wo_bytes;
  void *d_q = NULL, *d_k = NULL, *d_v = NULL, *d_refk = NULL, *d_refv = NULL, *d_wo = NULL;
  float* d_x = NULL;
  float* h_x = NULL;
  char name[256];
  cudaError_t e;

  if (argc != 14) {
    fprintf(stderr, "usage: %s DIR B H D F GRID_H GRID_W REF_FRAMES BOUNDARY_FRAMES REF_T CHUNKS STEPS SHIFT\n",
            argv[0]);
    return 2;
  }
  dir = argv[1];
  B = atoi(argv[2]);
  H = atoi(argv[3]);
  D = atoi(argv[4]);
  F = atoi(argv[5]);
  gh = atoi(argv[6]);
  gw = atoi(argv[7]);
  ref_frames = atoi(argv[8]);
  bnd_frames = atoi(argv[9]);
  ref_t = atoi(argv[10]);
  chunks = atoi(argv[11]);
  steps = atoi(argv[12]);
  shift = atof(argv[13]);
  if (steps < 1 || steps > 64 || chunks < 1) {
    fprintf(stderr, "steps must be in [1, 64] and chunks >= 1\n");
    return 2;
  }
  n_tok = (size_t)F * gh * gw;
  n_ref = (size_t)ref_frames * gh * gw;
  tok_bytes = (size_t)B * n_tok * H * D * 2;
  ref_bytes = (size_t)B * n_ref * H * D * 2;
  x_bytes = (size_t)B * n_tok * H * D * 4;
  wo_bytes = (size_t)H * D * H * D * 2;

  if ((rc = flow_time_grid(steps, shift, dt)) != SAVGB_OK) return fail_call("flow_time_grid", rc);

  if ((e = cudaMalloc(&d_q, tok_bytes)) != cudaSuccess || (e = cudaMalloc(&d_k, tok_bytes)) != cudaSuccess ||
      (e = cudaMalloc(&d_v, tok_bytes)) != cudaSuccess || (e = cudaMalloc(&d_refk, ref_bytes)) != cudaSuccess ||
      (e = cudaMalloc(&d_refv, ref_bytes)) != cudaSuccess || (e = cudaMalloc(&d_wo, wo_bytes)) != cudaSuccess ||
      (e = cudaMalloc((void**)&d_x, x_bytes)) != cudaSuccess)
    return fail_cuda("cudaMalloc", e);
  h_x = (float*)malloc(x_bytes);
  if (!h_x) return 1;
  if (upload(dir, "ref_k.bin", d_refk, ref_bytes) || upload(dir, "ref_v.bin", d_refv, ref_bytes) ||
      upload(dir, "w_o.bin", d_wo, wo_bytes))
    return 1;

  cfg.B = B;
  cfg.H = H;
  cfg.D = D;
  cfg.F = F;
  cfg.grid_h = gh;
  cfg.grid_w = gw;
  cfg.ref_frames = ref_frames;
  cfg.boundary_frames = bnd_frames;
  cfg.ref_t = ref_t;
  cfg.rope_base = 10000.0;
  cfg.softmax_scale = 0.f;
  cfg.interp_chunks = 0;
  cfg.qkv_block = 0;
  cfg.host_io = 0;
  cfg.exact_softmax = 0;
  /* the handle runs on the legacy default stream (NULL) */
  if ((rc = chunk_stream_create(&cfg, NULL, &s)) != SAVGB_OK) return fail_call("chunk_stream_create", rc);
  if ((rc = chunk_stream_set_reference(s, d_refk, d_refv)) != SAVGB_OK)
    return fail_call("chunk_stream_set_reference", rc);

  for (c = 0; c < chunks; ++c) {
    snprintf(name, sizeof name, "x_%d.bin", c);
    /* the previous chunk's steps have finished: chunk_stream_sync below */
    if (upload(dir, name, d_x, x_bytes)) return 1;
    for (st = 0; st < steps; ++st) {
      /* a step's q, k, v buffers are overwritten only after the previous
       * step has finished reading them */
      if ((e = cudaDeviceSynchronize()) != cudaSuccess) return fail_cuda("cudaDeviceSynchronize", e);
      snprintf(name, sizeof name, "q_%d_%d.bin", c, st);
      if (upload(dir, name, d_q, tok_bytes)) return 1;
      snprintf(name, sizeof name, "k_%d_%d.bin", c, st);
      if (upload(dir, name, d_k, tok_bytes)) return 1;
      snprintf(name, sizeof name, "v_%d_%d.bin", c, st);
      if (upload(dir, name, d_v, tok_bytes)) return 1;
      rc = chunk_stream_step(s, d_q, d_k, d_v, d_wo, NULL, d_x, (float)dt[st], st == steps - 1);
      if (rc != SAVGB_OK) return fail_call("chunk_stream_step", rc);
    }
    if ((rc = chunk_stream_end_chunk(s)) != SAVGB_OK) return fail_call("chunk_stream_end_chunk", rc);
    if ((rc = chunk_stream_sync(s)) != SAVGB_OK) return fail_call("chunk_stream_sync", rc);
    if ((e = cudaMemcpy(h_x, d_x, x_bytes, cudaMemcpyDeviceToHost)) != cudaSuccess)
      return fail_cuda("cudaMemcpy (read-back)", e);
    snprintf(name, sizeof name, "out_%d.bin", c);
    if (write_file(dir, name, h_x, x_bytes)) {
      fprintf(stderr, "cannot write %s\n", name);
      return 1;
    }
  }
  if ((rc = chunk_stream_destroy(s)) != SAVGB_OK) return fail_call("chunk_stream_destroy", rc);
  cudaFree(d_q);
  cudaFree(d_k);
  cudaFree(d_v);
  cudaFree(d_refk);
  cudaFree(d_refv);
  cudaFree(d_wo);
  cudaFree(d_x);
  free(h_x);
  printf("ok\n");
  return 0;
}
