/*
 * Drives a layerwise mixed-width job through libob's C ABI from plain C --
 * device memory from the CUDA runtime, no Python, no torch -- with the
 * method's schedules taken from the library alone: a 1-bit group
 * (ob_plan_step says when to call ob_reset_errors, then ob_step), a 2-bit
 * group and an FP16 group (ob_codec_step, which applies the reset, the
 * FP16 send period and the per-width Philox key itself).  The ctxs are
 * configured with reset_interval = 3, send_period = 2 and seed = 1234.
 *
 * The oracle's side below states the same schedules on its own (reset
 * before compressed steps 4 and 7, FP16 exchanged on even steps, 2-bit
 * key 1234 + 2) and runs the oracle's C functions.  After each of 7
 * compressed steps every group's parameters must be bit-identical.  Exit
 * status 0 on success.
 *
 * Build (the test does this): nvcc -O2 -I include c_abi_mixed.c -L<libob dir>
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
void orc_compress_worker(const struct orc_layout* L, const uint64_t* layer_off, uint64_t nl,
                         const float* sigma, const float* rho, float b1, const float* g,
                         const float* m, float* e, uint32_t* bits, float* scales,
                         float* x_out);
void orc_server_reduce(const struct orc_layout* L, const uint64_t* layer_off, uint64_t nl,
                       const float* rho, const uint32_t* bits, const float* scales,
                       float* e_s, uint32_t* sbits, float* sscales, float* y_out);
void orc_adam_update(const struct orc_layout* L, const uint32_t* sbits, const float* sscales,
                     const float* v, float eps, float lr, float* m, float* p);
void orc_qb_compress_worker(const struct orc_layout* L, int bits, float b1, float clip,
                            uint64_t w, uint64_t seed, uint64_t step, const float* g,
                            const float* m, float* e, uint32_t* codes, float* bscales);
void orc_qb_server(const struct orc_layout* L, int bits, uint64_t seed, uint64_t step,
                   const uint32_t* codes, const float* bscales, float* e_s, uint32_t* scodes,
                   float* sbscales);
void orc_qb_adam_at(const struct orc_layout* L, int bits, float eps, float lr, uint64_t k0,
                    uint64_t len, const uint32_t* scodes, const float* sbscales, const float* v,
                    float* m, float* p);
void orc_f16_compress_worker(const struct orc_layout* L, float b1, float clip, int send,
                             const float* g, const float* m, float* e, uint16_t* h);
void orc_f16_server(const struct orc_layout* L, const uint16_t* h, float* e_s, uint16_t* hs);
void orc_f16_adam(const struct orc_layout* L, int send, float eps, float lr, const uint16_t* hs,
                  const float* v, float* m, float* p);

enum { NW = 3, STEPS = 7 };

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
      exit(2);                                                               \
    }                                                                        \
  } while (0)
#define OK(ctx, x)                                                           \
  do {                                                                       \
    ob_status s_ = (x);                                                      \
    if (s_ != OB_OK) {                                                       \
      fprintf(stderr, "%s: status %d: %s\n", #x, s_, ob_last_error(ctx));   \
      exit(3);                                                               \
    }                                                                        \
  } while (0)

/* One group: its ctx and device buffers, and the oracle's host state. */
struct group {
  int bits;
  size_t n, np, words, nc;
  ob_ctx* ctx;
  struct orc_layout L;
  float *d_g[NW], *d_err[NW], *d_m, *d_v, *d_p, *d_es, *d_sc, *d_ssc;
  void *d_msg, *d_smsg, *d_ws;
  float *g[NW], *e[NW], *m, *v, *p, *es, *sc, *ssc;
  void *msg, *smsg;
};

static float* dalloc(size_t bytes) {
  void* p = NULL;
  CK(cudaMalloc(&p, bytes));
  CK(cudaMemset(p, 0, bytes));
  return (float*)p;
}

static void setup(struct group* G, int bits, size_t n) {
  ob_config cfg;
  memset(&cfg, 0, sizeof cfg);
  cfg.n = n;
  cfg.W = NW;
  cfg.chunk = 2048;
  cfg.align = bits == 1 ? 32 : 256;
  cfg.grad_dtype = OB_GRAD_F32;
  cfg.b1 = 0.9f;
  cfg.b2 = 0.999f;
  cfg.eps = 1e-8f;
  cfg.lr = 1e-4f;
  cfg.reset_interval = 3;
  cfg.send_period = 2;
  cfg.seed = 1234;
  G->bits = bits;
  G->n = n;
  ob_ctx* ctx = NULL;
  OK(ctx, ob_init(&cfg, &ctx));
  G->ctx = ctx;
  ob_layout lay;
  OK(ctx, ob_get_layout(ctx, &lay));
  orc_make_layout(n, NW, cfg.align, cfg.chunk, &G->L);
  if (G->L.n_pad != lay.n_pad) {
    fprintf(stderr, "layouts differ\n");
    exit(4);
  }
  G->np = lay.n_pad;
  G->nc = lay.n_chunks;
  size_t msg_bytes, smsg_bytes, sc_count = 0;
  if (bits == 1) {
    G->words = lay.words_per_worker;
    msg_bytes = (size_t)NW * G->words * 4;
    smsg_bytes = G->words * 4;
    sc_count = G->nc;
  } else if (bits == 16) {
    msg_bytes = (size_t)NW * G->np * 2;
    smsg_bytes = G->np * 2;
  } else {
    size_t nblk = 0;
    OK(ctx, ob_qb_sizes(ctx, bits, &G->words, &nblk));
    msg_bytes = (size_t)NW * G->words * 4;
    smsg_bytes = G->words * 4;
    sc_count = nblk;
  }
  for (int w = 0; w < NW; ++w) {
    G->d_g[w] = dalloc(G->np * 4);
    G->d_err[w] = dalloc(G->np * 4);
    G->g[w] = (float*)calloc(G->np, 4);
    G->e[w] = (float*)calloc(G->np, 4);
  }
  G->d_m = dalloc(G->np * 4);
  G->d_v = dalloc(G->np * 4);
  G->d_p = dalloc(G->np * 4);
  G->d_es = dalloc(G->np * 4);
  G->d_msg = dalloc(msg_bytes);
  G->d_smsg = dalloc(smsg_bytes);
  G->d_sc = sc_count ? dalloc((size_t)NW * sc_count * 4) : NULL;
  G->d_ssc = sc_count ? dalloc(sc_count * 4) : NULL;
  G->m = (float*)calloc(G->np, 4);
  G->v = (float*)calloc(G->np, 4);
  G->p = (float*)calloc(G->np, 4);
  G->es = (float*)calloc(G->np, 4);
  G->msg = calloc(msg_bytes, 1);
  G->smsg = calloc(smsg_bytes, 1);
  G->sc = (float*)calloc((size_t)NW * (sc_count ? sc_count : 1), 4);
  G->ssc = (float*)calloc(sc_count ? sc_count : 1, 4);
  size_t ws = 0;
  OK(ctx, ob_workspace_bytes(ctx, &ws));
  G->d_ws = dalloc(ws);
  OK(ctx, ob_set_workspace(ctx, G->d_ws, ws, 0));
  for (size_t k = 0; k < n; ++k) {
    G->p[k] = uniform_pm(0.02f);
    G->v[k] = 1e-6f + uniform_pm(5e-7f);
    G->m[k] = uniform_pm(1e-3f);
  }
  CK(cudaMemcpy(G->d_p, G->p, G->np * 4, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(G->d_v, G->v, G->np * 4, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(G->d_m, G->m, G->np * 4, cudaMemcpyHostToDevice));
  if (bits == 1)
    OK(ctx, ob_begin_compression(ctx, G->d_err, G->d_es, (uint32_t*)G->d_msg, G->d_sc,
                                 (uint32_t*)G->d_smsg, G->d_ssc, NULL, NULL, NULL, NULL, 1, 0));
  else
    OK(ctx, ob_zero_errors(ctx, G->d_err, G->d_es, 0));
}

/* The library's side of compressed step t: the schedule comes from libob. */
static void library_step(struct group* G, uint64_t t) {
  ob_ctx* ctx = G->ctx;
  const void* gp[NW];
  for (int w = 0; w < NW; ++w) gp[w] = G->d_g[w];
  if (G->bits == 1) {
    ob_plan plan;
    OK(ctx, ob_plan_step(ctx, 1, t, &plan));
    if (plan.reset)
      OK(ctx, ob_reset_errors(ctx, G->d_err, (const uint32_t*)G->d_msg, G->d_sc, G->d_es,
                              (const uint32_t*)G->d_smsg, G->d_ssc, 0));
    OK(ctx, ob_step(ctx, gp, G->d_m, G->d_err, (uint32_t*)G->d_msg, G->d_sc, G->d_es,
                    (uint32_t*)G->d_smsg, G->d_ssc, G->d_v, NULL, G->d_p, NULL, 0));
  } else {
    OK(ctx, ob_codec_step(ctx, G->bits, t, gp, G->d_m, G->d_err, G->d_msg, G->d_sc, G->d_es,
                          G->d_smsg, G->d_ssc, G->d_v, G->d_p, 0));
  }
}

/* The oracle's side, with the schedules stated here independently. */
static void oracle_step(struct group* G, uint64_t t) {
  const struct orc_layout* L = &G->L;
  if (t > 1 && (t - 1) % 3 == 0) { /* reset_interval = 3 */
    for (int w = 0; w < NW; ++w) memset(G->e[w], 0, G->np * 4);
    memset(G->es, 0, G->np * 4);
  }
  if (G->bits == 1) {
    const size_t ow = (G->np + 31) / 32;
    uint32_t* bits = (uint32_t*)G->msg;
    for (int w = 0; w < NW; ++w)
      orc_compress_worker(L, NULL, 0, NULL, NULL, 0.9f, G->g[w], G->m, G->e[w], bits + w * ow,
                          G->sc + w * G->nc, NULL);
    orc_server_reduce(L, NULL, 0, NULL, bits, G->sc, G->es, (uint32_t*)G->smsg, G->ssc, NULL);
    orc_adam_update(L, (uint32_t*)G->smsg, G->ssc, G->v, 1e-8f, 1e-4f, G->m, G->p);
  } else if (G->bits == 16) {
    const int send = t % 2 == 0; /* send_period = 2 */
    uint16_t* h = (uint16_t*)G->msg;
    for (int w = 0; w < NW; ++w)
      orc_f16_compress_worker(L, 0.9f, 0.0f, send, G->g[w], G->m, G->e[w], h + w * G->np);
    if (send) orc_f16_server(L, h, G->es, (uint16_t*)G->smsg);
    orc_f16_adam(L, send, 1e-8f, 1e-4f, (uint16_t*)G->smsg, G->v, G->m, G->p);
  } else {
    const uint64_t key = 1234 + (uint64_t)G->bits; /* seed + bits */
    const size_t nblk = G->np / 256;
    uint32_t* codes = (uint32_t*)G->msg;
    for (int w = 0; w < NW; ++w)
      orc_qb_compress_worker(L, G->bits, 0.9f, 0.0f, (uint64_t)w, key, t, G->g[w], G->m, G->e[w],
                             codes + w * G->words, G->sc + w * nblk);
    orc_qb_server(L, G->bits, key, t, codes, G->sc, G->es, (uint32_t*)G->smsg, G->ssc);
    orc_qb_adam_at(L, G->bits, 1e-8f, 1e-4f, 0, G->np, (uint32_t*)G->smsg, G->ssc, G->v, G->m,
                   G->p);
  }
}

int main(void) {
  struct group groups[3];
  setup(&groups[0], 1, 9001);
  setup(&groups[1], 2, 20000);
  setup(&groups[2], 16, 3001);
  int failures = 0;
  float* back = (float*)calloc(20480, 4);
  for (uint64_t t = 1; t <= STEPS; ++t) {
    for (int i = 0; i < 3; ++i) {
      struct group* G = &groups[i];
      for (int w = 0; w < NW; ++w) {
        for (size_t k = 0; k < G->n; ++k) G->g[w][k] = uniform_pm(1e-3f);
        CK(cudaMemcpy(G->d_g[w], G->g[w], G->np * 4, cudaMemcpyHostToDevice));
      }
      library_step(G, t);
      oracle_step(G, t);
      CK(cudaMemcpy(back, G->d_p, G->n * 4, cudaMemcpyDeviceToHost));
      if (memcmp(back, G->p, G->n * 4) != 0) {
        fprintf(stderr, "step %d: parameters of the %d-bit group differ\n", (int)t, G->bits);
        ++failures;
      }
    }
  }
  for (int i = 0; i < 3; ++i) {
    unsigned code = 0;
    OK(groups[i].ctx, ob_device_error(groups[i].ctx, &code, 0));
    failures += code != 0;
    OK(groups[i].ctx, ob_destroy(groups[i].ctx));
  }
  printf(failures ? "FAILED (%d)\n" : "c abi mixed ok\n", failures);
  return failures ? 1 : 0;
}
