/*
 * Drives one simulated 1-bit Adam job through libob's C ABI from plain C --
 * device memory from the CUDA runtime, no Python, no torch -- and checks it
 * step by step against the oracle's C functions (test infrastructure):
 * 2 warmup steps, the start of compression, 3 compressed steps.  After
 * every step the parameters, the server's sign words and its chunk scales
 * must be bit-identical.  Exit status 0 on success.
 *
 * Build (the test does this): nvcc -O2 -I include c_abi_step.c -L<libob dir>
 *   -lob -L<oracle dir> -loracle -Xlinker -rpath,<both dirs>
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "ob.h"

/* The oracle's C entry points (oracle/oracle.cpp). */
struct orc_layout {
  uint64_t n, W, A, C, P, n_pad, cpp, nc;
};
int orc_make_layout(uint64_t n, uint64_t W, uint64_t A, uint64_t C, struct orc_layout* out);
void orc_warmup_step(const struct orc_layout* L, const uint64_t* layer_off, uint64_t nl,
                     const float* const* grads, int mode, float b1, float b2, float eps,
                     float lr, float c_min, float c_max, float* m, float* v, float* p,
                     float* c_sum, float* c_out);
void orc_compress_worker(const struct orc_layout* L, const uint64_t* layer_off, uint64_t nl,
                         const float* sigma, const float* rho, float b1, const float* g,
                         const float* m, float* e, uint32_t* bits, float* scales,
                         float* x_out);
void orc_server_reduce(const struct orc_layout* L, const uint64_t* layer_off, uint64_t nl,
                       const float* rho, const uint32_t* bits, const float* scales,
                       float* e_s, uint32_t* sbits, float* sscales, float* y_out);
void orc_adam_update(const struct orc_layout* L, const uint32_t* sbits, const float* sscales,
                     const float* v, float eps, float lr, float* m, float* p);

enum { NW = 4 }; /* workers */
#define N 10037u

static uint32_t rng = 2463534242u;
static float uniform_pm(float scale) { /* xorshift32, uniform in [-scale, scale) */
  rng ^= rng << 13;
  rng ^= rng >> 17;
  rng ^= rng << 5;
  return scale * ((float)(rng >> 8) * (1.0f / 8388608.0f) - 1.0f);
}

#define CK(x)                                                                \
  do {                                                                       \
    cudaError_t e_ = (x);                                                    \
    if (e_ != cudaSuccess) {                                                 \
      fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));               \
      return 2;                                                              \
    }                                                                        \
  } while (0)
#define OK(x)                                                                \
  do {                                                                       \
    ob_status s_ = (x);                                                      \
    if (s_ != OB_OK) {                                                       \
      fprintf(stderr, "%s: status %d: %s\n", #x, s_, ob_last_error(ctx));   \
      return 3;                                                              \
    }                                                                        \
  } while (0)

int main(void) {
  ob_config cfg;
  memset(&cfg, 0, sizeof cfg);
  cfg.n = N;
  cfg.W = NW;
  cfg.chunk = 4096;
  cfg.align = 32;
  cfg.grad_dtype = OB_GRAD_F32;
  cfg.b1 = 0.9f;
  cfg.b2 = 0.999f;
  cfg.eps = 1e-8f;
  cfg.lr = 1e-4f;
  cfg.r_thr = 0.1f;
  cfg.r_min = 0.5f;
  cfg.r_max = 4.0f;
  cfg.c_min = 0.01f;
  cfg.c_max = 10.0f;
  ob_ctx* ctx = NULL;
  OK(ob_init(&cfg, &ctx));
  ob_layout lay;
  OK(ob_get_layout(ctx, &lay));
  struct orc_layout L;
  if (orc_make_layout(N, NW, 32, 4096, &L) != 0 || L.n_pad != lay.n_pad || L.nc != lay.n_chunks) {
    fprintf(stderr, "layouts differ\n");
    return 4;
  }
  const size_t np = lay.n_pad, words = lay.words_per_worker, nc = lay.n_chunks;
  const size_t owords = (np + 31) / 32; /* the oracle's rows are not rounded up */

  /* device buffers */
  float *d_g[NW], *d_err[NW], *d_m, *d_v, *d_p, *d_es, *d_scales, *d_sscales;
  uint32_t *d_bits, *d_sbits;
  void* d_ws;
  size_t ws_bytes = 0;
  for (int w = 0; w < NW; ++w) {
    CK(cudaMalloc((void**)&d_g[w], np * 4));
    CK(cudaMalloc((void**)&d_err[w], np * 4));
  }
  CK(cudaMalloc((void**)&d_m, np * 4));
  CK(cudaMalloc((void**)&d_v, np * 4));
  CK(cudaMalloc((void**)&d_p, np * 4));
  CK(cudaMalloc((void**)&d_es, np * 4));
  CK(cudaMalloc((void**)&d_bits, (size_t)NW * words * 4));
  CK(cudaMalloc((void**)&d_scales, (size_t)NW * nc * 4));
  CK(cudaMalloc((void**)&d_sbits, words * 4));
  CK(cudaMalloc((void**)&d_sscales, nc * 4));
  OK(ob_workspace_bytes(ctx, &ws_bytes));
  CK(cudaMalloc(&d_ws, ws_bytes));
  OK(ob_set_workspace(ctx, d_ws, ws_bytes, 0));

  /* host state of the oracle */
  float *g[NW], *e[NW];
  for (int w = 0; w < NW; ++w) {
    g[w] = (float*)calloc(np, 4);
    e[w] = (float*)calloc(np, 4);
  }
  float* m = (float*)calloc(np, 4);
  float* v = (float*)calloc(np, 4);
  float* p = (float*)calloc(np, 4);
  float* es = (float*)calloc(np, 4);
  uint32_t* bits = (uint32_t*)calloc((size_t)NW * owords, 4);
  float* scales = (float*)calloc((size_t)NW * nc, 4);
  uint32_t* sbits = (uint32_t*)calloc(owords, 4);
  float* sscales = (float*)calloc(nc, 4);
  float* back = (float*)calloc(np, 4);
  uint32_t* wback = (uint32_t*)calloc(words, 4);
  for (size_t k = 0; k < N; ++k) p[k] = uniform_pm(0.02f);
  CK(cudaMemset(d_m, 0, np * 4));
  CK(cudaMemset(d_v, 0, np * 4));
  CK(cudaMemcpy(d_p, p, np * 4, cudaMemcpyHostToDevice));

  const void* gp[NW];
  const float* hg[NW];
  for (int w = 0; w < NW; ++w) {
    gp[w] = d_g[w];
    hg[w] = g[w];
  }
  int failures = 0;
  for (int step = 0; step < 5; ++step) {
    for (int w = 0; w < NW; ++w) {
      for (size_t k = 0; k < N; ++k) g[w][k] = uniform_pm(1e-3f);
      CK(cudaMemcpy(d_g[w], g[w], np * 4, cudaMemcpyHostToDevice));
    }
    if (step < 2) {
      OK(ob_warmup_step(ctx, gp, d_m, d_v, d_p, OB_MODE_ADAM, NULL, 0));
      orc_warmup_step(&L, NULL, 0, hg, 0, cfg.b1, cfg.b2, cfg.eps, cfg.lr, 0.0f, 0.0f, m, v, p,
                      NULL, NULL);
    } else {
      if (step == 2) {
        OK(ob_begin_compression(ctx, d_err, d_es, d_bits, d_scales, d_sbits, d_sscales, NULL,
                                NULL, NULL, NULL, 2, 0));
        for (int w = 0; w < NW; ++w) memset(e[w], 0, np * 4);
        memset(es, 0, np * 4);
      }
      OK(ob_step(ctx, gp, d_m, d_err, d_bits, d_scales, d_es, d_sbits, d_sscales, d_v, NULL,
                 d_p, NULL, 0));
      for (int w = 0; w < NW; ++w)
        orc_compress_worker(&L, NULL, 0, NULL, NULL, cfg.b1, g[w], m, e[w], bits + w * owords,
                            scales + w * nc, NULL);
      orc_server_reduce(&L, NULL, 0, NULL, bits, scales, es, sbits, sscales, NULL);
      orc_adam_update(&L, sbits, sscales, v, cfg.eps, cfg.lr, m, p);
      CK(cudaMemcpy(wback, d_sbits, words * 4, cudaMemcpyDeviceToHost));
      if (memcmp(wback, sbits, owords * 4) != 0) {
        fprintf(stderr, "step %d: server sign words differ\n", step);
        ++failures;
      }
      CK(cudaMemcpy(back, d_sscales, nc * 4, cudaMemcpyDeviceToHost));
      if (memcmp(back, sscales, nc * 4) != 0) {
        fprintf(stderr, "step %d: server scales differ\n", step);
        ++failures;
      }
    }
    CK(cudaMemcpy(back, d_p, np * 4, cudaMemcpyDeviceToHost));
    if (memcmp(back, p, N * 4) != 0) {
      fprintf(stderr, "step %d: parameters differ\n", step);
      ++failures;
    }
  }
  unsigned code = 0;
  OK(ob_device_error(ctx, &code, 0));
  if (code != 0) {
    fprintf(stderr, "device error word %u\n", code);
    ++failures;
  }
  OK(ob_destroy(ctx));
  printf(failures ? "FAILED (%d)\n" : "c abi ok\n", failures);
  return failures ? 1 : 0;
}
