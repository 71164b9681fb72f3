/*
 * A plain C user of libgbln: allocates device memory with the CUDA runtime,
 * runs RMSNorm forward + backward (+ dW finalize), RoPE forward + backward,
 * SwiGLU forward + backward, LayerNorm forward + backward (+ dW/dB finalize)
 * and the MXFP8 RMSNorm forward through the C ABI on one stream, and writes
 * every input and output (as float32) to a binary file that the test compares
 * with the CPU oracle.  Inputs come from a fixed linear congruential generator.
 *
 * usage: gbln_client OUT.bin
 * exit status: 0 on success, 2 on a CUDA error, 3 on a library error.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "gbln.h"

enum { T = 37, H = 96, HQ = 3, HK = 1, D = 32, I = 200, MAXPOS = 64 };

static uint64_t lcg_state = 12345;
static float lcg_uniform(void) { /* in [-1, 1) */
  lcg_state = lcg_state * 6364136223846793005ULL + 1442695040888963407ULL;
  return (float)((lcg_state >> 40) & 0xFFFFFF) / 8388608.0f - 1.0f;
}

#define CK(x)                                                              \
  do {                                                                     \
    cudaError_t e_ = (x);                                                  \
    if (e_ != cudaSuccess) {                                               \
      fprintf(stderr, "CUDA error %s at line %d\n", cudaGetErrorString(e_), __LINE__); \
      exit(2);                                                             \
    }                                                                      \
  } while (0)
#define GK(x)                                                              \
  do {                                                                     \
    int s_ = (int)(x);                                                     \
    if (s_ != GBLN_OK) {                                                   \
      fprintf(stderr, "gbln error %s at line %d\n", gbln_status_string(s_), __LINE__); \
      exit(3);                                                             \
    }                                                                      \
  } while (0)

static float* dev_alloc(size_t n) {
  void* p = NULL;
  CK(cudaMalloc(&p, n * sizeof(float)));
  return (float*)p;
}
static float* dev_from(const float* h, size_t n) {
  float* d = dev_alloc(n);
  CK(cudaMemcpy(d, h, n * sizeof(float), cudaMemcpyHostToDevice));
  return d;
}
static void dump(FILE* f, const char* name, const float* d, size_t n, int from_device) {
  float* h = (float*)malloc(n * sizeof(float));
  if (from_device) CK(cudaMemcpy(h, d, n * sizeof(float), cudaMemcpyDeviceToHost));
  else memcpy(h, d, n * sizeof(float));
  uint32_t len = (uint32_t)strlen(name), cnt = (uint32_t)n;
  fwrite(&len, 4, 1, f);
  fwrite(name, 1, len, f);
  fwrite(&cnt, 4, 1, f);
  fwrite(h, sizeof(float), n, f);
  free(h);
}
static float* host_rand(size_t n, float scale, float shift) {
  float* h = (float*)malloc(n * sizeof(float));
  for (size_t i = 0; i < n; ++i) h[i] = shift + scale * lcg_uniform();
  return h;
}

int main(int argc, char** argv) {
  if (argc != 2) {
    fprintf(stderr, "usage: %s OUT.bin\n", argv[0]);
    return 1;
  }
  if (gbln_version() < 100) return 3;
  cudaStream_t stream;
  CK(cudaStreamCreate(&stream));
  gbln_stream_t s = (gbln_stream_t)stream;

  /* inputs */
  float *x = host_rand(T * H, 2.f, 0.f), *r = host_rand(T * H, 2.f, 0.f), *w = host_rand(H, 0.2f, 1.f);
  float *dy = host_rand(T * H, 1.f, 0.f), *dres = host_rand(T * H, 1.f, 0.f);
  float *q = host_rand(T * HQ * D, 1.f, 0.f), *k = host_rand(T * HK * D, 1.f, 0.f);
  float *gate = host_rand(T * I, 3.f, 0.f), *up = host_rand(T * I, 1.f, 0.f), *dout = host_rand(T * I, 1.f, 0.f);
  int32_t cu[3] = {0, 20, T};
  float eps = 1e-5f;
  double theta = 10000.0;

  float *dx_ = dev_from(x, T * H), *dr_ = dev_from(r, T * H), *dw_ = dev_from(w, H);
  float *y = dev_alloc(T * H), *hres = dev_alloc(T * H), *rstd = dev_alloc(T);
  float *ddy = dev_from(dy, T * H), *ddres = dev_from(dres, T * H), *dxo = dev_alloc(T * H);
  GK(gbln_rmsnorm_fwd(dx_, dr_, dw_, y, hres, rstd, T, H, eps, GBLN_F32, GBLN_F32, s));
  int64_t P = gbln_rmsnorm_bwd_num_partials(T, H, GBLN_F32);
  if (P < 1) return 3;
  float *part = dev_alloc((size_t)P * H), *dW = dev_alloc(H);
  GK(gbln_rmsnorm_bwd(ddy, ddres, hres, dw_, rstd, dxo, part, P, T, H, GBLN_F32, GBLN_F32, s));
  GK(gbln_rmsnorm_dw_finalize(part, P, H, dW, 0, s));

  int32_t* dcu = NULL;
  int32_t* dpos = NULL;
  CK(cudaMalloc((void**)&dcu, sizeof(cu)));
  CK(cudaMalloc((void**)&dpos, T * sizeof(int32_t)));
  CK(cudaMemcpy(dcu, cu, sizeof(cu), cudaMemcpyHostToDevice));
  float *table = dev_alloc((size_t)MAXPOS * D), *dq = dev_from(q, T * HQ * D), *dk = dev_from(k, T * HK * D);
  float *qo = dev_alloc(T * HQ * D), *ko = dev_alloc(T * HK * D), *qb = dev_alloc(T * HQ * D), *kb = dev_alloc(T * HK * D);
  GK(gbln_positions_from_cu_seqlens(dcu, 2, dpos, T, s));
  GK(gbln_rope_table(table, MAXPOS, D, theta, s));
  GK(gbln_rope_fwd(dq, dk, qo, ko, dpos, table, MAXPOS, T, HQ, HK, D, GBLN_F32, s));
  GK(gbln_rope_bwd(dq, dk, qb, kb, dpos, table, MAXPOS, T, HQ, HK, D, GBLN_F32, s));

  float *dg = dev_from(gate, T * I), *du = dev_from(up, T * I), *ddo = dev_from(dout, T * I);
  float *so = dev_alloc(T * I), *sdg = dev_alloc(T * I), *sdu = dev_alloc(T * I);
  GK(gbln_swiglu_fwd(dg, du, so, T, I, GBLN_F32, s));
  GK(gbln_swiglu_bwd(ddo, dg, du, sdg, sdu, T, I, GBLN_F32, s));
  /* LayerNorm (residual + bias) on the same rows, and the MXFP8 RMSNorm forward */
  float *bias = host_rand(H, 1.f, 0.f), *dbias = dev_from(bias, H);
  float *ly = dev_alloc(T * H), *lh = dev_alloc(T * H), *lmean = dev_alloc(T), *lrstd = dev_alloc(T);
  float *ldx = dev_alloc(T * H);
  GK(gbln_layernorm_fwd(dx_, dr_, dw_, dbias, ly, lh, lmean, lrstd, T, H, eps, GBLN_F32, GBLN_F32, s));
  int64_t LP = gbln_layernorm_bwd_num_partials(T, H, GBLN_F32);
  if (LP < 1) return 3;
  float *lpart = dev_alloc((size_t)LP * 2 * H), *ldW = dev_alloc(H), *ldB = dev_alloc(H);
  GK(gbln_layernorm_bwd(ddy, ddres, lh, dw_, lmean, lrstd, ldx, lpart, LP, T, H, GBLN_F32, GBLN_F32, s));
  GK(gbln_layernorm_dwdb_finalize(lpart, LP, H, ldW, ldB, 0, s));
  uint8_t *q8 = NULL, *sc8 = NULL;
  float *mh = dev_alloc(T * H), *mrstd = dev_alloc(T);
  CK(cudaMalloc((void**)&q8, T * H));
  CK(cudaMalloc((void**)&sc8, T * (H / 32)));
  GK(gbln_rmsnorm_fwd_mxfp8(dx_, dr_, dw_, NULL, q8, sc8, mh, mrstd, T, H, eps, GBLN_F32, GBLN_F32, s));
  CK(cudaStreamSynchronize(stream));

  uint32_t err = 0;
  GK(gbln_device_error(&err, 0));
  if (err) return 3;

  FILE* f = fopen(argv[1], "wb");
  if (!f) return 1;
  dump(f, "x", x, T * H, 0); dump(f, "residual", r, T * H, 0); dump(f, "weight", w, H, 0);
  dump(f, "dy", dy, T * H, 0); dump(f, "dres", dres, T * H, 0);
  dump(f, "y", y, T * H, 1); dump(f, "h", hres, T * H, 1); dump(f, "rstd", rstd, T, 1);
  dump(f, "dx", dxo, T * H, 1); dump(f, "dW", dW, H, 1);
  dump(f, "q", q, T * HQ * D, 0); dump(f, "k", k, T * HK * D, 0);
  dump(f, "q_out", qo, T * HQ * D, 1); dump(f, "k_out", ko, T * HK * D, 1);
  dump(f, "dq_in", qb, T * HQ * D, 1); dump(f, "dk_in", kb, T * HK * D, 1);
  dump(f, "gate", gate, T * I, 0); dump(f, "up", up, T * I, 0); dump(f, "dout", dout, T * I, 0);
  dump(f, "out", so, T * I, 1); dump(f, "dgate", sdg, T * I, 1); dump(f, "dup", sdu, T * I, 1);
  dump(f, "bias", bias, H, 0);
  dump(f, "ln_y", ly, T * H, 1); dump(f, "ln_mean", lmean, T, 1); dump(f, "ln_rstd", lrstd, T, 1);
  dump(f, "ln_dx", ldx, T * H, 1); dump(f, "ln_dW", ldW, H, 1); dump(f, "ln_dB", ldB, H, 1);
  {
    uint8_t hq[T * H], hs[T * (H / 32)];
    float fq[T * H], fs[T * (H / 32)];
    CK(cudaMemcpy(hq, q8, sizeof(hq), cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(hs, sc8, sizeof(hs), cudaMemcpyDeviceToHost));
    for (int i = 0; i < T * H; ++i) fq[i] = (float)hq[i];
    for (int i = 0; i < T * (H / 32); ++i) fs[i] = (float)hs[i];
    dump(f, "y_e4m3", fq, T * H, 0);
    dump(f, "y_scale", fs, T * (H / 32), 0);
  }
  {
    int32_t hp[T];
    float fp[T];
    CK(cudaMemcpy(hp, dpos, sizeof(hp), cudaMemcpyDeviceToHost));
    for (int i = 0; i < T; ++i) fp[i] = (float)hp[i];
    dump(f, "positions", fp, T, 0);
  }
  fclose(f);
  printf("gbln_client ok\n");
  return 0;
}
