/*
 * Drives a simulated 1-bit LAMB job through libob's C ABI from plain C, with
 * the momentum held in sign form and the server output double-buffered
 * (ob_step_db), and checks it step by step against the oracle's C functions
 * (test infrastructure): 2 warmup steps, the start of compression, one
 * compressed step with the dense momentum from warmup, then 3 steps in
 * sign form, swapping the two server buffers after each.  Layers of odd
 * sizes (3000, 7, 7030) share the buffer; the gradient scale falls 3x per
 * compressed step, so r and c move.  After every step p, the server's sign
 * words and chunk scales and every layer's c must be bit-identical.  Exit
 * status 0 on success.
 *
 * Build (the test does this): nvcc -O2 -I include c_abi_lamb_signm.c
 *   -L<libob dir> -lob -L<oracle dir> -loracle -Xlinker -rpath,<both dirs>
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
void orc_lamb_begin(const struct orc_layout* L, const uint64_t* layer_off, uint64_t nl,
                    const float* m, const float* c_sum, uint64_t warmup_steps, float* s,
                    float* c_avg, float* r_prev, float* c_prev, float* c_prev2);
void orc_lamb_rho(uint64_t nl, const float* c_prev2, const float* c_prev, float* rho);
void orc_compress_worker(const struct orc_layout* L, const uint64_t* layer_off, uint64_t nl,
                         const float* sigma, const float* rho, float b1, const float* g,
                         const float* m, float* e, uint32_t* bits, float* scales,
                         float* x_out);
void orc_server_reduce(const struct orc_layout* L, const uint64_t* layer_off, uint64_t nl,
                       const float* rho, const uint32_t* bits, const float* scales,
                       float* e_s, uint32_t* sbits, float* sscales, float* y_out);
void orc_lamb_pass_a(const struct orc_layout* L, const uint64_t* layer_off, uint64_t nl,
                     const float* sigma, const uint32_t* sbits, const float* sscales,
                     const float* v_frozen, float b1, float b2, float* m, float* v_fresh,
                     float* R);
void orc_lamb_ratio(uint64_t nl, const float* R, float r_thr, float r_min, float r_max,
                    float c_min, float c_max, int frozen, const float* c_avg, float* r_prev,
                    float* c_prev, float* c_prev2, float* c_out);
void orc_lamb_pass_b(const struct orc_layout* L, const uint64_t* layer_off, uint64_t nl,
                     const float* c, const float* m, const float* v_frozen, float eps, float lr,
                     float* p);

enum { NW = 4, NL = 3 }; /* workers, layers */
#define N 10037u

static const size_t OFF[NL + 1] = {0, 3000, 3007, N};
static const float LAYER_STD[NL] = {3e-3f, 1e-2f, 5e-4f};

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

static float* dalloc(size_t count) {
  float* p = NULL;
  if (cudaMalloc((void**)&p, count * sizeof(float)) != cudaSuccess) return NULL;
  if (cudaMemset(p, 0, count * sizeof(float)) != cudaSuccess) return NULL;
  return p;
}

int main(void) {
  ob_config cfg;
  memset(&cfg, 0, sizeof cfg);
  cfg.n = N;
  cfg.W = NW;
  cfg.chunk = 2048;
  cfg.align = 32;
  cfg.grad_dtype = OB_GRAD_F32;
  cfg.n_layers = NL;
  cfg.layer_offsets = OFF;
  cfg.b1 = 0.9f;
  cfg.b2 = 0.999f;
  cfg.eps = 1e-6f;
  cfg.lr = 1e-3f;
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
  if (orc_make_layout(N, NW, 32, 2048, &L) != 0 || L.n_pad != lay.n_pad || L.nc != lay.n_chunks) {
    fprintf(stderr, "layouts differ\n");
    return 4;
  }
  uint64_t off64[NL + 1];
  for (int l = 0; l <= NL; ++l) off64[l] = OFF[l];
  const size_t np = lay.n_pad, words = lay.words_per_worker, nc = lay.n_chunks;
  const size_t owords = (np + 31) / 32; /* the oracle's rows are not rounded up */

  /* device buffers: two server buffer pairs (A, B) for the sign form */
  float *d_g[NW], *d_err[NW];
  for (int w = 0; w < NW; ++w) {
    if (!(d_g[w] = dalloc(np)) || !(d_err[w] = dalloc(np))) return 2;
  }
  float* d_m = dalloc(np);
  float* d_v = dalloc(np);
  float* d_vf = dalloc(np);
  float* d_p = dalloc(np);
  float* d_es = dalloc(np);
  float* d_scales = dalloc((size_t)NW * nc);
  float* d_ssc[2] = {dalloc(nc), dalloc(nc)};
  uint32_t* d_bits = (uint32_t*)dalloc((size_t)NW * words);
  uint32_t* d_sb[2] = {(uint32_t*)dalloc(words), (uint32_t*)dalloc(words)};
  float* d_ls = dalloc(7 * NL);
  if (!d_m || !d_v || !d_vf || !d_p || !d_es || !d_scales || !d_ssc[0] || !d_ssc[1] ||
      !d_bits || !d_sb[0] || !d_sb[1] || !d_ls)
    return 2;
  ob_layer_state ls = {d_ls, d_ls + NL, d_ls + 2 * NL, d_ls + 3 * NL,
                       d_ls + 4 * NL, d_ls + 5 * NL, d_ls + 6 * NL};
  void* d_ws;
  size_t ws_bytes = 0;
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
  float* vf = (float*)calloc(np, 4);
  float* p = (float*)calloc(np, 4);
  float* es = (float*)calloc(np, 4);
  uint32_t* bits = (uint32_t*)calloc((size_t)NW * owords, 4);
  float* scales = (float*)calloc((size_t)NW * nc, 4);
  uint32_t* sbits = (uint32_t*)calloc(owords, 4);
  float* sscales = (float*)calloc(nc, 4);
  float s[NL], c_avg[NL], r_prev[NL], c_prev[NL], c_prev2[NL], c_sum[NL], c_out[NL];
  float rho[NL], R[NL];
  memset(c_sum, 0, sizeof c_sum);
  float* back = (float*)calloc(np, 4);
  uint32_t* wback = (uint32_t*)calloc(words, 4);
  float lsback[NL];
  for (size_t k = 0; k < N; ++k) p[k] = uniform_pm(0.02f);
  CK(cudaMemcpy(d_p, p, np * 4, cudaMemcpyHostToDevice));

  const void* gp[NW];
  const float* hg[NW];
  for (int w = 0; w < NW; ++w) {
    gp[w] = d_g[w];
    hg[w] = g[w];
  }
  int failures = 0, cur = 0; /* cur: the server buffer holding the last output */
  float fall = 1.0f;
  for (int step = 0; step < 6; ++step) {
    for (int w = 0; w < NW; ++w) {
      for (int l = 0; l < NL; ++l)
        for (size_t k = OFF[l]; k < OFF[l + 1]; ++k) g[w][k] = uniform_pm(LAYER_STD[l] * fall);
      CK(cudaMemcpy(d_g[w], g[w], np * 4, cudaMemcpyHostToDevice));
    }
    if (step < 2) {
      OK(ob_warmup_step(ctx, gp, d_m, d_v, d_p, OB_MODE_LAMB, &ls, 0));
      orc_warmup_step(&L, off64, NL, hg, 1, cfg.b1, cfg.b2, cfg.eps, cfg.lr, cfg.c_min,
                      cfg.c_max, m, v, p, c_sum, c_out);
    } else {
      if (step == 2) {
        OK(ob_begin_compression(ctx, d_err, d_es, d_bits, d_scales, d_sb[0], d_ssc[0], d_m, d_v,
                                d_vf, &ls, 2, 0));
        for (int w = 0; w < NW; ++w) memset(e[w], 0, np * 4);
        memset(es, 0, np * 4);
        memcpy(vf, v, np * 4);
        orc_lamb_begin(&L, off64, NL, m, c_sum, 2, s, c_avg, r_prev, c_prev, c_prev2);
        /* the first compressed step takes the dense m from warmup */
        OK(ob_step(ctx, gp, d_m, d_err, d_bits, d_scales, d_es, d_sb[0], d_ssc[0], d_v, d_vf,
                   d_p, &ls, 0));
      } else {
        OK(ob_step_db(ctx, gp, d_err, d_bits, d_scales, d_es, d_sb[cur], d_ssc[cur],
                      d_sb[1 - cur], d_ssc[1 - cur], d_v, d_vf, d_p, &ls, 0));
        cur = 1 - cur;
      }
      orc_lamb_rho(NL, c_prev2, c_prev, rho);
      for (int w = 0; w < NW; ++w)
        orc_compress_worker(&L, off64, NL, s, rho, cfg.b1, g[w], m, e[w], bits + w * owords,
                            scales + w * nc, NULL);
      orc_server_reduce(&L, off64, NL, rho, bits, scales, es, sbits, sscales, NULL);
      memset(R, 0, sizeof R);
      orc_lamb_pass_a(&L, off64, NL, s, sbits, sscales, v, cfg.b1, cfg.b2, m, vf, R);
      orc_lamb_ratio(NL, R, cfg.r_thr, cfg.r_min, cfg.r_max, cfg.c_min, cfg.c_max, 0, c_avg,
                     r_prev, c_prev, c_prev2, c_out);
      orc_lamb_pass_b(&L, off64, NL, c_out, m, v, cfg.eps, cfg.lr, p);
      CK(cudaMemcpy(wback, d_sb[cur], words * 4, cudaMemcpyDeviceToHost));
      if (memcmp(wback, sbits, owords * 4) != 0) {
        fprintf(stderr, "step %d: server sign words differ\n", step);
        ++failures;
      }
      CK(cudaMemcpy(back, d_ssc[cur], nc * 4, cudaMemcpyDeviceToHost));
      if (memcmp(back, sscales, nc * 4) != 0) {
        fprintf(stderr, "step %d: server scales differ\n", step);
        ++failures;
      }
      CK(cudaMemcpy(lsback, ls.c_t, NL * 4, cudaMemcpyDeviceToHost));
      if (memcmp(lsback, c_out, NL * 4) != 0) {
        fprintf(stderr, "step %d: c differs\n", step);
        ++failures;
      }
      fall *= 1.0f / 3.0f;
    }
    CK(cudaMemcpy(back, d_p, np * 4, cudaMemcpyDeviceToHost));
    if (memcmp(back, p, N * 4) != 0) {
      fprintf(stderr, "step %d: parameters differ\n", step);
      ++failures;
    }
  }
  /* the dense momentum rebuilt from the signs equals the oracle's m */
  OK(ob_decompress(ctx, d_sb[cur], d_ssc[cur], &ls, d_m, 0));
  CK(cudaMemcpy(back, d_m, np * 4, cudaMemcpyDeviceToHost));
  if (memcmp(back, m, N * 4) != 0) {
    fprintf(stderr, "momentum rebuilt from the signs differs\n");
    ++failures;
  }
  CK(cudaMemcpy(lsback, ls.r_prev, NL * 4, cudaMemcpyDeviceToHost));
  int r_moved = 0;
  for (int l = 0; l < NL; ++l) r_moved |= lsback[l] != 1.0f;
  if (!r_moved) {
    fprintf(stderr, "r never moved: the run does not exercise the ratio\n");
    ++failures;
  }
  unsigned code = 0;
  OK(ob_device_error(ctx, &code, 0));
  if (code != 0) {
    fprintf(stderr, "device error word %u\n", code);
    ++failures;
  }
  OK(ob_destroy(ctx));
  printf(failures ? "FAILED (%d)\n" : "c abi lamb ok\n", failures);
  return failures ? 1 : 0;
}
