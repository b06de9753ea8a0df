// C entry points of the layerwise mixed-width codecs (b-bit blocks and
// FP16); declared in ob.h.  Host-side checks only; the arithmetic is in
// k_mixed.cu.
#include <cstdarg>
#include <cstdio>

#include "ob_internal.cuh"

namespace {

ob_status failf(ob_ctx* ctx, ob_status st, const char* fmt, ...) {
  char buf[400];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  return ob::ctx_fail(ctx, st, buf);
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

#define OB_MIX_PTR(ctx, ptr, al, name)                                                  \
  do {                                                                                  \
    if (!(ptr)) return failf(ctx, OB_ERR_INVALID, "%s is NULL", name);                  \
    if (!aligned((ptr), (al)))                                                          \
      return failf(ctx, OB_ERR_ALIGN, "%s is not %d-byte aligned", name, (int)(al));    \
  } while (0)

// The checks every codec call shares: a ctx whose partitions are whole
// blocks of 256, and (for the b-bit codec) a supported width.
ob_status check_ctx(ob_ctx* ctx, int bits) {
  if (!ctx) return ob::ctx_fail(nullptr, OB_ERR_INVALID, "ctx is NULL");
  const ob_config& c = *ob::ctx_config(ctx);
  if (c.align % 256 != 0)
    return failf(ctx, OB_ERR_UNSUPPORTED,
                 "mixed-width codecs need the alignment A = %zu to be a multiple of 256",
                 c.align);
  if (bits != 0 && bits != 2 && bits != 4 && bits != 8)
    return failf(ctx, OB_ERR_INVALID, "bits = %d must be 2, 4 or 8", bits);
  return OB_OK;
}

ob_status check_workers(ob_ctx* ctx, const void* const* grads, float* const* err) {
  const int W = ob::ctx_config(ctx)->W;
  if (grads) {
    for (int w = 0; w < W; ++w) OB_MIX_PTR(ctx, grads[w], 16, "grads[w]");
  } else {
    return failf(ctx, OB_ERR_INVALID, "grads is NULL");
  }
  if (!err) return failf(ctx, OB_ERR_INVALID, "err is NULL");
  for (int w = 0; w < W; ++w) OB_MIX_PTR(ctx, err[w], 16, "err[w]");
  return OB_OK;
}

ob_status device_sms(ob_ctx* ctx, int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return failf(ctx, OB_ERR_CUDA, "device query: %s", cudaGetErrorString(e));
  return OB_OK;
}

ob_status launched(ob_ctx* ctx, cudaError_t e, const char* what) {
  if (e != cudaSuccess) return failf(ctx, OB_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return OB_OK;
}

}  // namespace

extern "C" {

ob_status ob_qb_sizes(const ob_ctx* ctx, int bits, size_t* words_per_worker,
                      size_t* n_blocks) {
  OB_TRACE();
  ob_status st = check_ctx(const_cast<ob_ctx*>(ctx), bits);
  if (st) return st;
  if (bits == 0) return failf(const_cast<ob_ctx*>(ctx), OB_ERR_INVALID, "bits = 0");
  const ob::Geo& G = *ob::ctx_geo(ctx);
  if (words_per_worker) *words_per_worker = (size_t)(G.n_pad * (uint64_t)bits / 32);
  if (n_blocks) *n_blocks = (size_t)(G.n_pad / 256);
  return OB_OK;
}

ob_status ob_zero_errors(ob_ctx* ctx, float* const* err, float* err_s, ob_stream_t stream) {
  OB_TRACE();
  if (!ctx) return ob::ctx_fail(nullptr, OB_ERR_INVALID, "ctx is NULL");
  const ob::Geo& G = *ob::ctx_geo(ctx);
  if (!err) return failf(ctx, OB_ERR_INVALID, "err is NULL");
  for (uint32_t w = 0; w < G.W; ++w) OB_MIX_PTR(ctx, err[w], 16, "err[w]");
  OB_MIX_PTR(ctx, err_s, 16, "err_s");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  for (uint32_t w = 0; w < G.W && e == cudaSuccess; ++w)
    e = cudaMemsetAsync(err[w], 0, G.n_pad * sizeof(float), s);
  if (e == cudaSuccess) e = cudaMemsetAsync(err_s, 0, G.n_pad * sizeof(float), s);
  return launched(ctx, e, "zero_errors");
}

ob_status ob_compress_qb(ob_ctx* ctx, int bits, const void* const* grads, const float* m,
                         float* const* err, uint32_t* codes, float* bscales, uint64_t seed,
                         uint64_t step, ob_stream_t stream) {
  OB_TRACE();
  ob_status st = check_ctx(ctx, bits);
  if (st) return st;
  if (bits == 0) return failf(ctx, OB_ERR_INVALID, "bits = 0");
  if ((st = check_workers(ctx, grads, err))) return st;
  OB_MIX_PTR(ctx, m, 16, "m");
  OB_MIX_PTR(ctx, codes, 16, "codes");
  OB_MIX_PTR(ctx, bscales, 4, "bscales");
  int sms = 0;
  if ((st = device_sms(ctx, &sms))) return st;
  const ob::Geo& G = *ob::ctx_geo(ctx);
  const ob_config& c = *ob::ctx_config(ctx);
  ob::QbCompressArgs a{};
  for (uint32_t w = 0; w < G.W; ++w) {
    a.g[w] = grads[w];
    a.e[w] = err[w];
  }
  a.m = m;
  a.codes = codes;
  a.scales = bscales;
  a.n = G.n;
  a.n_pad = G.n_pad;
  a.row_words = G.n_pad * (uint64_t)bits / 32;
  a.seed = seed;
  a.step = step;
  a.W = G.W;
  a.b1 = c.b1;
  a.clip = c.clip_value;
  return launched(ctx,
                  ob::launch_qb_compress(a, bits, c.grad_dtype == OB_GRAD_BF16, sms,
                                         reinterpret_cast<cudaStream_t>(stream)),
                  "compress_qb");
}

ob_status ob_server_reduce_qb(ob_ctx* ctx, int bits, const uint32_t* codes,
                              const float* bscales, float* err_s, uint32_t* scodes,
                              float* sbscales, uint64_t seed, uint64_t step,
                              ob_stream_t stream) {
  OB_TRACE();
  ob_status st = check_ctx(ctx, bits);
  if (st) return st;
  if (bits == 0) return failf(ctx, OB_ERR_INVALID, "bits = 0");
  OB_MIX_PTR(ctx, codes, 16, "codes");
  OB_MIX_PTR(ctx, bscales, 4, "bscales");
  OB_MIX_PTR(ctx, err_s, 16, "err_s");
  OB_MIX_PTR(ctx, scodes, 16, "scodes");
  OB_MIX_PTR(ctx, sbscales, 4, "sbscales");
  int sms = 0;
  if ((st = device_sms(ctx, &sms))) return st;
  const ob::Geo& G = *ob::ctx_geo(ctx);
  ob::QbServerArgs a{};
  a.codes = codes;
  a.scales = bscales;
  a.e_s = err_s;
  a.scodes = scodes;
  a.sscales = sbscales;
  a.n = G.n;
  a.n_pad = G.n_pad;
  a.row_words = G.n_pad * (uint64_t)bits / 32;
  a.seed = seed;
  a.step = step;
  a.W = G.W;
  return launched(ctx,
                  ob::launch_qb_server(a, bits, sms, reinterpret_cast<cudaStream_t>(stream)),
                  "server_reduce_qb");
}

ob_status ob_adam_step_qb(ob_ctx* ctx, int bits, const uint32_t* scodes, const float* sbscales,
                          const float* v_frozen, float* m, float* p, ob_stream_t stream) {
  OB_TRACE();
  ob_status st = check_ctx(ctx, bits);
  if (st) return st;
  if (bits == 0) return failf(ctx, OB_ERR_INVALID, "bits = 0");
  OB_MIX_PTR(ctx, scodes, 16, "scodes");
  OB_MIX_PTR(ctx, sbscales, 4, "sbscales");
  OB_MIX_PTR(ctx, v_frozen, 16, "v_frozen");
  OB_MIX_PTR(ctx, m, 16, "m");
  OB_MIX_PTR(ctx, p, 16, "p");
  int sms = 0;
  if ((st = device_sms(ctx, &sms))) return st;
  const ob::Geo& G = *ob::ctx_geo(ctx);
  const ob_config& c = *ob::ctx_config(ctx);
  ob::QbUpdateArgs a{};
  a.scodes = scodes;
  a.sscales = sbscales;
  a.v = v_frozen;
  a.m = m;
  a.p = p;
  a.n = G.n;
  a.n_pad = G.n_pad;
  a.lr = c.lr;
  a.eps = c.eps;
  return launched(ctx, ob::launch_qb_adam(a, bits, sms, reinterpret_cast<cudaStream_t>(stream)),
                  "adam_step_qb");
}

ob_status ob_compress_f16(ob_ctx* ctx, int send, const void* const* grads, const float* m,
                          float* const* err, uint16_t* h, ob_stream_t stream) {
  OB_TRACE();
  ob_status st = check_ctx(ctx, 0);
  if (st) return st;
  if ((st = check_workers(ctx, grads, err))) return st;
  OB_MIX_PTR(ctx, m, 16, "m");
  if (send) OB_MIX_PTR(ctx, h, 16, "h");
  int sms = 0;
  if ((st = device_sms(ctx, &sms))) return st;
  const ob::Geo& G = *ob::ctx_geo(ctx);
  const ob_config& c = *ob::ctx_config(ctx);
  ob::F16Args a{};
  for (uint32_t w = 0; w < G.W; ++w) {
    a.g[w] = grads[w];
    a.e[w] = err[w];
  }
  a.m = const_cast<float*>(m);
  a.h = h;
  a.n = G.n;
  a.n_pad = G.n_pad;
  a.W = G.W;
  a.send = send ? 1 : 0;
  a.b1 = c.b1;
  a.clip = c.clip_value;
  return launched(ctx,
                  ob::launch_f16_compress(a, c.grad_dtype == OB_GRAD_BF16, sms,
                                          reinterpret_cast<cudaStream_t>(stream)),
                  "compress_f16");
}

ob_status ob_server_reduce_f16(ob_ctx* ctx, const uint16_t* h, float* err_s, uint16_t* hs,
                               ob_stream_t stream) {
  OB_TRACE();
  ob_status st = check_ctx(ctx, 0);
  if (st) return st;
  OB_MIX_PTR(ctx, h, 16, "h");
  OB_MIX_PTR(ctx, err_s, 16, "err_s");
  OB_MIX_PTR(ctx, hs, 16, "hs");
  int sms = 0;
  if ((st = device_sms(ctx, &sms))) return st;
  const ob::Geo& G = *ob::ctx_geo(ctx);
  ob::F16Args a{};
  a.h = const_cast<uint16_t*>(h);
  a.hs = hs;
  a.e_s = err_s;
  a.n = G.n;
  a.n_pad = G.n_pad;
  a.W = G.W;
  return launched(ctx,
                  ob::launch_f16_server(a, sms, reinterpret_cast<cudaStream_t>(stream)),
                  "server_reduce_f16");
}

ob_status ob_adam_step_f16(ob_ctx* ctx, int send, const uint16_t* hs, const float* v_frozen,
                           float* m, float* p, ob_stream_t stream) {
  OB_TRACE();
  ob_status st = check_ctx(ctx, 0);
  if (st) return st;
  OB_MIX_PTR(ctx, m, 16, "m");
  if (send) {
    OB_MIX_PTR(ctx, hs, 16, "hs");
    OB_MIX_PTR(ctx, v_frozen, 16, "v_frozen");
    OB_MIX_PTR(ctx, p, 16, "p");
  }
  int sms = 0;
  if ((st = device_sms(ctx, &sms))) return st;
  const ob::Geo& G = *ob::ctx_geo(ctx);
  const ob_config& c = *ob::ctx_config(ctx);
  ob::F16Args a{};
  a.hs = const_cast<uint16_t*>(hs);
  a.v = v_frozen;
  a.m = m;
  a.p = p;
  a.n = G.n;
  a.n_pad = G.n_pad;
  a.W = G.W;
  a.send = send ? 1 : 0;
  a.lr = c.lr;
  a.eps = c.eps;
  return launched(ctx, ob::launch_f16_adam(a, sms, reinterpret_cast<cudaStream_t>(stream)),
                  "adam_step_f16");
}

ob_status ob_plan_step(const ob_ctx* ctx, int bits, uint64_t t, ob_plan* out) {
  OB_TRACE();
  if (!ctx || !out) return ob::ctx_fail(nullptr, OB_ERR_INVALID, "ctx or out is NULL");
  ob_ctx* c = const_cast<ob_ctx*>(ctx);
  if (bits != 1 && bits != 2 && bits != 4 && bits != 8 && bits != 16)
    return failf(c, OB_ERR_INVALID, "bits = %d must be 1, 2, 4, 8 or 16", bits);
  if (t < 1) return failf(c, OB_ERR_INVALID, "t = 0: compressed steps count from 1");
  const ob_config& cfg = *ob::ctx_config(ctx);
  ob_plan pl{};
  // the periodic reset of the "1bit Adam" write-up, section 4.1
  pl.reset = cfg.reset_interval > 0 && t > 1 && (t - 1) % cfg.reset_interval == 0;
  // the FP16 group is exchanged every send_period-th step (section 3.2 table)
  const uint64_t period = cfg.send_period > 1 ? cfg.send_period : 1;
  pl.send = bits == 16 ? (t % period == 0) : 1;
  // one Philox stream per width (section 6, layerwise_bits)
  pl.key = (bits == 2 || bits == 4 || bits == 8) ? cfg.seed + (uint64_t)bits : 0;
  pl.step = t;
  *out = pl;
  return OB_OK;
}

ob_status ob_codec_step(ob_ctx* ctx, int bits, uint64_t t, const void* const* grads, float* m,
                        float* const* err, void* msg, float* msg_scales, float* err_s,
                        void* smsg, float* smsg_scales, const float* v_frozen, float* p,
                        ob_stream_t stream) {
  OB_TRACE();
  if (!ctx) return ob::ctx_fail(nullptr, OB_ERR_INVALID, "ctx is NULL");
  if (bits == 1) return failf(ctx, OB_ERR_INVALID, "bits = 1: use the 1-bit calls");
  ob_plan pl;
  ob_status st = ob_plan_step(ctx, bits, t, &pl);
  if (st) return st;
  if (pl.reset && (st = ob_zero_errors(ctx, err, err_s, stream))) return st;
  if (bits == 16) {
    uint16_t* h = static_cast<uint16_t*>(msg);
    uint16_t* hs = static_cast<uint16_t*>(smsg);
    if ((st = ob_compress_f16(ctx, pl.send, grads, m, err, h, stream))) return st;
    if (pl.send && (st = ob_server_reduce_f16(ctx, h, err_s, hs, stream))) return st;
    return ob_adam_step_f16(ctx, pl.send, hs, v_frozen, m, p, stream);
  }
  uint32_t* codes = static_cast<uint32_t*>(msg);
  uint32_t* scodes = static_cast<uint32_t*>(smsg);
  if ((st = ob_compress_qb(ctx, bits, grads, m, err, codes, msg_scales, pl.key, pl.step,
                           stream)))
    return st;
  if ((st = ob_server_reduce_qb(ctx, bits, codes, msg_scales, err_s, scodes, smsg_scales,
                                pl.key, pl.step, stream)))
    return st;
  return ob_adam_step_qb(ctx, bits, scodes, smsg_scales, v_frozen, m, p, stream);
}

}  // extern "C"
