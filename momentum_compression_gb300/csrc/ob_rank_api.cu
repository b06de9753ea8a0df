// C entry points of one rank of a multi-process job (one worker and one
// server per process; declared in ob.h): the 1-bit LAMB summary's 3-phase
// exchange (paragraphs 2 and 4: local compression, an all-to-all of the
// compressed chunks, the server's average and re-compression, an
// all-gather of the result) with the collectives left to the caller.
//
// ob_compress_worker compresses the rank's own worker into the same row
// layout as ob_compress, so partition j's words and scales are contiguous
// blocks: the all-to-all sends block j to rank j unchanged.
// ob_server_reduce_part reduces one partition from the W received blocks;
// the all-gather of its outputs, in rank order, is the whole server output
// of ob_server_reduce.  Both run the same kernels as the resident path.
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

#define OB_RANK_PTR(ctx, ptr, al, name)                                                 \
  do {                                                                                  \
    if (!(ptr)) return failf(ctx, OB_ERR_INVALID, "%s is NULL", name);                  \
    if (!aligned((ptr), (al)))                                                          \
      return failf(ctx, OB_ERR_ALIGN, "%s is not %d-byte aligned", name, (int)(al));    \
  } while (0)

ob_status ready(ob_ctx* ctx) {
  if (!ctx) return ob::ctx_fail(nullptr, OB_ERR_INVALID, "ctx is NULL");
  if (!ob::ctx_ws(ctx)) return failf(ctx, OB_ERR_STATE, "no workspace: call ob_set_workspace first");
  return OB_OK;
}

ob_status check_ls(ob_ctx* ctx, const ob_layer_state* ls) {
  const float* arr[] = {ls->s, ls->c_avg, ls->r_prev, ls->c_prev, ls->c_prev2, ls->c_t};
  for (const float* a : arr) OB_RANK_PTR(ctx, a, 4, "a layer-state array");
  return OB_OK;
}

ob_status launched(ob_ctx* ctx, cudaError_t e, const char* what) {
  if (e != cudaSuccess) return failf(ctx, OB_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return OB_OK;
}

}  // namespace

extern "C" {

ob_status ob_compress_worker(ob_ctx* ctx, const void* grad, const float* m,
                             const uint32_t* msbits, const float* msscales, float* err,
                             uint32_t* bits_row, float* scales_row, const ob_layer_state* ls,
                             ob_stream_t stream) {
  OB_TRACE();
  ob_status st = ready(ctx);
  if (st) return st;
  const ob::Geo& G = *ob::ctx_geo(ctx);
  const ob_config& cfg = *ob::ctx_config(ctx);
  OB_RANK_PTR(ctx, grad, 16, "grad");
  OB_RANK_PTR(ctx, err, 16, "err");
  OB_RANK_PTR(ctx, bits_row, 16, "bits_row");
  OB_RANK_PTR(ctx, scales_row, 4, "scales_row");
  const bool sign_form = m == nullptr;
  if (sign_form) {
    OB_RANK_PTR(ctx, msbits, 16, "msbits");
    OB_RANK_PTR(ctx, msscales, 4, "msscales");
  } else {
    OB_RANK_PTR(ctx, m, 16, "m");
    if (msbits || msscales)
      return failf(ctx, OB_ERR_INVALID, "give either m or (msbits, msscales), not both");
  }
  if (ls && (st = check_ls(ctx, ls))) return st;
  ob::CompressArgs a{};
  a.geo = G;
  a.ws = *ob::ctx_ws(ctx);
  a.nw = 1;
  a.g[0] = grad;
  a.e[0] = err;
  a.m = m;
  a.msbits = msbits;
  a.msscales = msscales;
  a.bits = bits_row;
  a.scales = scales_row;
  if (ls) {
    a.s = ls->s;
    a.c_prev = ls->c_prev;
    a.c_prev2 = ls->c_prev2;
  }
  a.ratio_ef = (cfg.flags & OB_FLAG_NO_RATIO_EF) ? 0 : 1;
  a.b1 = cfg.b1;
  a.ob1 = 1.0f - cfg.b1;
  a.clip = cfg.clip_value;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool bf16 = cfg.grad_dtype == OB_GRAD_BF16;
  const int sms = ob::ctx_sms(ctx);
  cudaError_t e = sign_form ? ob::launch_compress_signm(a, bf16, ls != nullptr, sms, s)
                            : ob::launch_compress(a, bf16, ls != nullptr, sms, s);
  if ((st = launched(ctx, e, "compress_worker"))) return st;
  return launched(ctx, ob::launch_finalize_scales(G, a.ws.wpart, 1, scales_row, sms, s),
                  "compress_worker: chunk scales");
}

ob_status ob_server_reduce_part(ob_ctx* ctx, int j, const uint32_t* recv_bits,
                                const float* recv_scales, float* err_s_part,
                                uint32_t* sbits_part, float* sscales_part,
                                const ob_layer_state* ls, ob_stream_t stream) {
  OB_TRACE();
  ob_status st = ready(ctx);
  if (st) return st;
  const ob::Geo& G = *ob::ctx_geo(ctx);
  const ob_config& cfg = *ob::ctx_config(ctx);
  if (j < 0 || (uint32_t)j >= G.W)
    return failf(ctx, OB_ERR_INVALID, "partition %d is not in [0, W = %u)", j, G.W);
  if (G.P % 128 != 0)
    return failf(ctx, OB_ERR_UNSUPPORTED,
                 "per-partition server calls need the partition size P = %llu to be a "
                 "multiple of 128 (alignment A a multiple of 128)",
                 (unsigned long long)G.P);
  OB_RANK_PTR(ctx, recv_bits, 16, "recv_bits");
  OB_RANK_PTR(ctx, recv_scales, 4, "recv_scales");
  OB_RANK_PTR(ctx, err_s_part, 16, "err_s_part");
  OB_RANK_PTR(ctx, sbits_part, 16, "sbits_part");
  OB_RANK_PTR(ctx, sscales_part, 4, "sscales_part");
  if (ls && (st = check_ls(ctx, ls))) return st;
  ob::ServerArgs a{};
  a.geo = G;
  a.ws = *ob::ctx_ws(ctx);
  a.T0 = (uint32_t)j * G.tpp;
  a.T1 = a.T0 + G.tpp;
  a.g0 = (uint32_t)j * G.cpp;
  a.base = (uint64_t)j * G.P;
  a.bits_stride = G.P / 32;
  a.sc_stride = G.cpp;
  a.bits = recv_bits;
  a.scales = recv_scales;
  a.e_s = err_s_part;
  a.sbits = sbits_part;
  a.sscales = sscales_part;
  a.sbits_old = sbits_part;
  a.sscales_old = sscales_part;
  if (ls) {
    a.c_prev = ls->c_prev;
    a.c_prev2 = ls->c_prev2;
  }
  a.ratio_ef = (cfg.flags & OB_FLAG_NO_RATIO_EF) ? 0 : 1;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int sms = ob::ctx_sms(ctx);
  if ((st = launched(ctx, ob::launch_server(a, ls != nullptr, sms, s), "server_reduce_part")))
    return st;
  return launched(ctx,
                  ob::launch_finalize_scales_range(G, a.ws.spart, 1, a.g0, G.cpp, sscales_part,
                                                   sms, s),
                  "server_reduce_part: chunk scales");
}

ob_status ob_reset_errors_rank(ob_ctx* ctx, int j, float* err, const uint32_t* bits_row,
                               const float* scales_row, float* err_s_part,
                               const uint32_t* sbits_part, const float* sscales_part,
                               ob_stream_t stream) {
  OB_TRACE();
  if (!ctx) return ob::ctx_fail(nullptr, OB_ERR_INVALID, "ctx is NULL");
  const ob::Geo& G = *ob::ctx_geo(ctx);
  if (j < 0 || (uint32_t)j >= G.W)
    return failf(ctx, OB_ERR_INVALID, "partition %d is not in [0, W = %u)", j, G.W);
  OB_RANK_PTR(ctx, err, 16, "err");
  OB_RANK_PTR(ctx, bits_row, 16, "bits_row");
  OB_RANK_PTR(ctx, scales_row, 4, "scales_row");
  OB_RANK_PTR(ctx, err_s_part, 16, "err_s_part");
  OB_RANK_PTR(ctx, sbits_part, 16, "sbits_part");
  OB_RANK_PTR(ctx, sscales_part, 4, "sscales_part");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int sms = ob::ctx_sms(ctx);
  ob::MaterializeArgs a{};
  a.geo = G;
  // the rank's own worker row, every tile
  a.nw = 1;
  a.T1 = G.n_tiles;
  a.e[0] = err;
  a.bits = bits_row;
  a.scales = scales_row;
  ob_status st = launched(ctx, ob::launch_reset_errors(a, sms, s), "reset_errors_rank: worker");
  if (st) return st;
  // its server partition: partition j's tiles, indexed from the partition
  ob::MaterializeArgs b{};
  b.geo = G;
  b.nw = 0;
  b.T0 = (uint32_t)j * G.tpp;
  b.T1 = b.T0 + G.tpp;
  b.g0 = (uint32_t)j * G.cpp;
  b.base = (uint64_t)j * G.P;
  b.e_s = err_s_part;
  b.sbits = sbits_part;
  b.sscales = sscales_part;
  return launched(ctx, ob::launch_reset_errors(b, sms, s), "reset_errors_rank: server");
}

}  // extern "C"
