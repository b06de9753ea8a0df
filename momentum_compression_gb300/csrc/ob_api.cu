// The C ABI of libob (include/ob.h): configuration checks, the layout of
// the fused buffer, the workspace, and the order of launches of each call.
// No device memory is allocated here; every buffer belongs to the caller.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "ob_internal.cuh"

using ob::Geo;
using ob::kTile;

struct ob_ctx {
  ob_config cfg{};
  std::vector<uint64_t> off;         // L+1 layer offsets
  std::vector<uint32_t> tile_layer;  // n_tiles
  std::vector<uint32_t> ltile_pref;  // L+1
  Geo geo{};
  ob_layout lay{};
  void* ws_base = nullptr;
  size_t ws_bytes = 0;
  ob::Workspace ws{};
  int sms = 0;
  std::string err;
};

namespace {

thread_local std::string g_err;

ob_status fail(ob_ctx* ctx, ob_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  if (ctx) ctx->err = buf;
  g_err = buf;
  return st;
}

ob_status cuda_fail(ob_ctx* ctx, cudaError_t e, const char* what) {
  return fail(ctx, OB_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

uint64_t cdiv(uint64_t a, uint64_t b) { return (a + b - 1) / b; }

size_t region(size_t& cursor, size_t bytes) {
  size_t at = cursor;
  cursor += (bytes + 255) / 256 * 256;
  return at;
}

struct Regions {
  size_t wpart, spart, tile_layer, layer_off, ltile_pref, lpart, Rbits, rms, gcnt, err, total;
};

Regions regions_of(const Geo& G) {
  Regions r{};
  size_t c = 0;
  r.wpart = region(c, (size_t)G.W * G.nc * G.tpc * sizeof(float));
  r.spart = region(c, (size_t)G.nc * G.tpc * sizeof(float));
  r.tile_layer = region(c, (size_t)G.n_tiles * sizeof(uint32_t));
  r.layer_off = region(c, (size_t)(G.L + 1) * sizeof(uint64_t));
  r.ltile_pref = region(c, (size_t)(G.L + 1) * sizeof(uint32_t));
  r.lpart = region(c, (size_t)2 * G.n_ltiles * sizeof(float));
  r.Rbits = region(c, (size_t)G.L * sizeof(unsigned));
  r.rms = region(c, (size_t)G.L * sizeof(float));
  r.gcnt = region(c, 4 * sizeof(unsigned));
  r.err = region(c, sizeof(unsigned));
  r.total = c;
  return r;
}

// Common checks of every call that runs kernels of a ctx.
ob_status ready(ob_ctx* ctx) {
  if (!ctx) return fail(nullptr, OB_ERR_INVALID, "ctx is NULL");
  if (!ctx->ws_base) return fail(ctx, OB_ERR_STATE, "no workspace: call ob_set_workspace first");
  return OB_OK;
}

#define OB_CHECK_PTR(ctx, ptr, align, name)                                             \
  do {                                                                                  \
    if (!(ptr)) return fail(ctx, OB_ERR_INVALID, "%s is NULL", name);                   \
    if (!aligned((ptr), (align)))                                                       \
      return fail(ctx, OB_ERR_ALIGN, "%s is not %d-byte aligned", name, (int)(align));  \
  } while (0)

ob_status check_grads(ob_ctx* ctx, const void* const* grads) {
  if (!grads) return fail(ctx, OB_ERR_INVALID, "grads is NULL");
  for (int w = 0; w < ctx->cfg.W; ++w) {
    if (!grads[w]) return fail(ctx, OB_ERR_INVALID, "grads[%d] is NULL", w);
    if (!aligned(grads[w], 16)) return fail(ctx, OB_ERR_ALIGN, "grads[%d] is not 16-byte aligned", w);
  }
  return OB_OK;
}

ob_status check_errs(ob_ctx* ctx, float* const* err) {
  if (!err) return fail(ctx, OB_ERR_INVALID, "err is NULL");
  for (int w = 0; w < ctx->cfg.W; ++w) {
    if (!err[w]) return fail(ctx, OB_ERR_INVALID, "err[%d] is NULL", w);
    if (!aligned(err[w], 16)) return fail(ctx, OB_ERR_ALIGN, "err[%d] is not 16-byte aligned", w);
  }
  return OB_OK;
}

ob_status check_ls(ob_ctx* ctx, const ob_layer_state* ls, bool need_sum) {
  if (!ls) return fail(ctx, OB_ERR_INVALID, "layer state is NULL");
  const float* arr[] = {ls->s, ls->c_avg, ls->r_prev, ls->c_prev, ls->c_prev2, ls->c_t};
  const char* nm[] = {"ls.s", "ls.c_avg", "ls.r_prev", "ls.c_prev", "ls.c_prev2", "ls.c_t"};
  for (int i = 0; i < 6; ++i) OB_CHECK_PTR(ctx, arr[i], 4, nm[i]);
  if (need_sum) OB_CHECK_PTR(ctx, ls->c_sum, 4, "ls.c_sum");
  return OB_OK;
}

ob_status launched(ob_ctx* ctx, cudaError_t e, const char* what) {
  if (e != cudaSuccess) return cuda_fail(ctx, e, what);
  return OB_OK;
}

}  // namespace

namespace ob {

// Read-only views of a ctx and its error slot, for the other translation
// units of the library.
const Geo* ctx_geo(const ob_ctx* ctx) { return &ctx->geo; }
const Workspace* ctx_ws(const ob_ctx* ctx) { return ctx->ws_base ? &ctx->ws : nullptr; }
int ctx_sms(const ob_ctx* ctx) { return ctx->sms; }
const ob_config* ctx_config(const ob_ctx* ctx) { return &ctx->cfg; }
ob_status ctx_fail(ob_ctx* ctx, ob_status st, const char* msg) {
  return fail(ctx, st, "%s", msg);
}

}  // namespace ob

extern "C" {

const char* ob_last_error(const ob_ctx* ctx) {
  OB_TRACE();
  return ctx ? ctx->err.c_str() : g_err.c_str();
}

ob_status ob_init(const ob_config* cfg, ob_ctx** out) {
  OB_TRACE();
  if (!cfg || !out) return fail(nullptr, OB_ERR_INVALID, "cfg or out is NULL");
  *out = nullptr;
  const ob_config& c = *cfg;
  if (c.n < 1 || c.n >= (1ull << 34))
    return fail(nullptr, OB_ERR_INVALID, "n = %zu must be in [1, 2^34)", c.n);
  if (c.W < 1) return fail(nullptr, OB_ERR_INVALID, "W = %d must be >= 1", c.W);
  if (c.W > OB_MAX_WORKERS)
    return fail(nullptr, OB_ERR_UNSUPPORTED, "W = %d exceeds %d", c.W, OB_MAX_WORKERS);
  if (c.chunk < 32 || c.chunk % 32)
    return fail(nullptr, OB_ERR_INVALID, "chunk = %zu must be a positive multiple of 32", c.chunk);
  if (c.align < 32 || c.align % 32)
    return fail(nullptr, OB_ERR_INVALID, "align = %zu must be a positive multiple of 32", c.align);
  if (c.grad_dtype != OB_GRAD_F32 && c.grad_dtype != OB_GRAD_BF16)
    return fail(nullptr, OB_ERR_INVALID, "grad_dtype = %d", c.grad_dtype);
  if (!(c.b1 >= 0.0f && c.b1 < 1.0f) || !(c.b2 >= 0.0f && c.b2 < 1.0f))
    return fail(nullptr, OB_ERR_INVALID, "betas must be in [0, 1)");
  if (!(c.eps >= 0.0f) || !(c.lr == c.lr))
    return fail(nullptr, OB_ERR_INVALID, "eps must be >= 0 and lr a number");
  if (c.n_layers < 0) return fail(nullptr, OB_ERR_INVALID, "n_layers < 0");
  if (!(c.clip_value >= 0.0f)) return fail(nullptr, OB_ERR_INVALID, "clip_value must be >= 0");

  ob_ctx* ctx = new ob_ctx();
  ctx->cfg = c;
  const uint32_t L = c.n_layers ? (uint32_t)c.n_layers : 1u;
  ctx->off.resize(L + 1);
  if (c.n_layers) {
    if (!c.layer_offsets) {
      delete ctx;
      return fail(nullptr, OB_ERR_INVALID, "layer_offsets is NULL");
    }
    for (uint32_t l = 0; l <= L; ++l) ctx->off[l] = c.layer_offsets[l];
    bool ok = ctx->off[0] == 0 && ctx->off[L] == c.n;
    for (uint32_t l = 0; l < L && ok; ++l) ok = ctx->off[l] < ctx->off[l + 1];
    if (!ok) {
      delete ctx;
      return fail(nullptr, OB_ERR_INVALID,
                  "layer_offsets must rise strictly from 0 to n = %zu", c.n);
    }
  } else {
    ctx->off[0] = 0;
    ctx->off[1] = c.n;
  }
  ctx->cfg.layer_offsets = nullptr;

  Geo& G = ctx->geo;
  const uint64_t W = (uint64_t)c.W;
  G.n = c.n;
  G.W = (uint32_t)W;
  G.P = cdiv(cdiv(c.n, W), c.align) * c.align;
  G.C = std::min<uint64_t>(c.chunk, G.P);
  const uint64_t cpp = cdiv(G.P, G.C);
  G.Cl = G.P - (cpp - 1) * G.C;
  G.n_pad = W * G.P;
  G.words = cdiv(G.n_pad / 32, 4) * 4;  // 16-byte aligned rows
  const uint64_t tpc = cdiv(G.C, kTile), tpl = cdiv(G.Cl, kTile);
  const uint64_t tpp = (cpp - 1) * tpc + tpl;
  const uint64_t n_tiles = W * tpp, nc = W * cpp;
  if (n_tiles >= (1ull << 31) || nc >= (1ull << 31)) {
    delete ctx;
    return fail(nullptr, OB_ERR_UNSUPPORTED, "too many tiles");
  }
  G.cpp = (uint32_t)cpp;
  G.tpc = (uint32_t)tpc;
  G.tpl = (uint32_t)tpl;
  G.tpp = (uint32_t)tpp;
  G.nc = (uint32_t)nc;
  G.n_tiles = (uint32_t)n_tiles;
  G.L = L;

  // Per-layer tile counts (tiles counted from each layer's start).
  ctx->ltile_pref.resize(L + 1);
  uint64_t acc = 0;
  for (uint32_t l = 0; l < L; ++l) {
    ctx->ltile_pref[l] = (uint32_t)acc;
    acc += cdiv(ctx->off[l + 1] - ctx->off[l], kTile);
  }
  ctx->ltile_pref[L] = (uint32_t)acc;
  if (acc >= (1ull << 31)) {
    delete ctx;
    return fail(nullptr, OB_ERR_UNSUPPORTED, "too many layer tiles");
  }
  G.n_ltiles = (uint32_t)acc;

  // Layer of each tile's first element.
  ctx->tile_layer.resize(n_tiles);
  for (uint64_t T = 0; T < n_tiles; ++T) {
    uint64_t j = T / tpp, r = T - j * tpp, kc = r / tpc, t = r - kc * tpc;
    uint64_t start = j * G.P + kc * G.C + t * kTile;
    uint64_t k = std::min<uint64_t>(start, c.n - 1);
    uint32_t l = (uint32_t)(std::upper_bound(ctx->off.begin(), ctx->off.end(), k) -
                            ctx->off.begin()) - 1;
    ctx->tile_layer[T] = std::min(l, L - 1);
  }

  ob_layout& lay = ctx->lay;
  lay.n = c.n;
  lay.n_pad = G.n_pad;
  lay.P = G.P;
  lay.chunk = G.C;
  lay.chunks_per_partition = cpp;
  lay.n_chunks = nc;
  lay.words_per_worker = G.words;
  lay.n_tiles = n_tiles;
  lay.W = c.W;
  lay.n_layers = (int)L;
  *out = ctx;
  return OB_OK;
}

ob_status ob_destroy(ob_ctx* ctx) {
  OB_TRACE();
  delete ctx;
  return OB_OK;
}

ob_status ob_get_layout(const ob_ctx* ctx, ob_layout* out) {
  OB_TRACE();
  if (!ctx || !out) return fail(nullptr, OB_ERR_INVALID, "ctx or out is NULL");
  *out = ctx->lay;
  return OB_OK;
}

ob_status ob_workspace_bytes(const ob_ctx* ctx, size_t* bytes) {
  OB_TRACE();
  if (!ctx || !bytes) return fail(nullptr, OB_ERR_INVALID, "ctx or bytes is NULL");
  *bytes = regions_of(ctx->geo).total;
  return OB_OK;
}

ob_status ob_set_workspace(ob_ctx* ctx, void* workspace, size_t bytes, ob_stream_t stream) {
  OB_TRACE();
  if (!ctx) return fail(nullptr, OB_ERR_INVALID, "ctx is NULL");
  const Regions r = regions_of(ctx->geo);
  if (!workspace) return fail(ctx, OB_ERR_INVALID, "workspace is NULL");
  if (!aligned(workspace, 256)) return fail(ctx, OB_ERR_ALIGN, "workspace is not 256-byte aligned");
  if (bytes < r.total)
    return fail(ctx, OB_ERR_INVALID, "workspace has %zu bytes, needs %zu", bytes, r.total);
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "device query");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* b = static_cast<char*>(workspace);
  e = cudaMemsetAsync(b, 0, r.total, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(b + r.tile_layer, ctx->tile_layer.data(),
                        ctx->tile_layer.size() * sizeof(uint32_t), cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(b + r.layer_off, ctx->off.data(), ctx->off.size() * sizeof(uint64_t),
                        cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(b + r.ltile_pref, ctx->ltile_pref.data(),
                        ctx->ltile_pref.size() * sizeof(uint32_t), cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "workspace initialisation");
  ob::Workspace& w = ctx->ws;
  w.wpart = reinterpret_cast<float*>(b + r.wpart);
  w.spart = reinterpret_cast<float*>(b + r.spart);
  w.tile_layer = reinterpret_cast<uint32_t*>(b + r.tile_layer);
  w.layer_off = reinterpret_cast<uint64_t*>(b + r.layer_off);
  w.ltile_pref = reinterpret_cast<uint32_t*>(b + r.ltile_pref);
  w.lpart = reinterpret_cast<float*>(b + r.lpart);
  w.Rbits = reinterpret_cast<unsigned*>(b + r.Rbits);
  w.rms = reinterpret_cast<float*>(b + r.rms);
  w.gcnt = reinterpret_cast<unsigned*>(b + r.gcnt);
  w.err = reinterpret_cast<unsigned*>(b + r.err);
  ctx->ws_base = workspace;
  ctx->ws_bytes = bytes;
  ctx->sms = sms;
  return OB_OK;
}

ob_status ob_warmup_step(ob_ctx* ctx, const void* const* grads, float* m, float* v, float* p,
                         int mode, const ob_layer_state* ls, ob_stream_t stream) {
  OB_TRACE();
  ob_status st = ready(ctx);
  if (st) return st;
  if (mode != OB_MODE_ADAM && mode != OB_MODE_LAMB)
    return fail(ctx, OB_ERR_INVALID, "mode = %d", mode);
  if ((st = check_grads(ctx, grads))) return st;
  OB_CHECK_PTR(ctx, m, 16, "m");
  OB_CHECK_PTR(ctx, v, 16, "v");
  OB_CHECK_PTR(ctx, p, 16, "p");
  if (mode == OB_MODE_LAMB && (st = check_ls(ctx, ls, true))) return st;
  ob::WarmupArgs a{};
  a.geo = ctx->geo;
  a.ws = ctx->ws;
  for (int w = 0; w < ctx->cfg.W; ++w) a.g[w] = grads[w];
  a.m = m;
  a.v = v;
  a.p = p;
  if (ls) a.ls = *ls;
  const ob_config& c = ctx->cfg;
  a.b1 = c.b1;
  a.ob1 = 1.0f - c.b1;
  a.b2 = c.b2;
  a.ob2 = 1.0f - c.b2;
  a.eps = c.eps;
  a.lr = c.lr;
  a.c_min = c.c_min;
  a.c_max = c.c_max;
  a.fW = (float)c.W;
  a.inv_w = ob::inv_workers((uint32_t)c.W);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool bf16 = c.grad_dtype == OB_GRAD_BF16;
  if (mode == OB_MODE_ADAM) return launched(ctx, ob::launch_warmup_adam(a, bf16, ctx->sms, s), "warmup");
  return launched(ctx, ob::launch_warmup_lamb(a, bf16, ctx->sms, s), "warmup");
}

ob_status ob_begin_compression(ob_ctx* ctx, float* const* err, float* err_s, uint32_t* bits,
                               float* scales, uint32_t* sbits, float* sscales, const float* m,
                               const float* v, float* v_fresh, const ob_layer_state* ls,
                               int warmup_steps, ob_stream_t stream) {
  OB_TRACE();
  ob_status st = ready(ctx);
  if (st) return st;
  const Geo& G = ctx->geo;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  // All six error and sign buffers NULL: a rank of a multi-process job
  // clears its own slices; only the LAMB part below runs.
  const bool none = !err && !err_s && !bits && !scales && !sbits && !sscales;
  if (!none) {
    if ((st = check_errs(ctx, err))) return st;
    OB_CHECK_PTR(ctx, err_s, 16, "err_s");
    OB_CHECK_PTR(ctx, bits, 16, "bits");
    OB_CHECK_PTR(ctx, scales, 4, "scales");
    OB_CHECK_PTR(ctx, sbits, 16, "sbits");
    OB_CHECK_PTR(ctx, sscales, 4, "sscales");
    for (uint32_t w = 0; w < G.W && e == cudaSuccess; ++w)
      e = cudaMemsetAsync(err[w], 0, G.n_pad * sizeof(float), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(err_s, 0, G.n_pad * sizeof(float), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(bits, 0, (size_t)G.W * G.words * sizeof(uint32_t), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(scales, 0, (size_t)G.W * G.nc * sizeof(float), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(sbits, 0, (size_t)G.words * sizeof(uint32_t), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(sscales, 0, (size_t)G.nc * sizeof(float), s);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "begin_compression: clearing the errors");
  }
  if (!ls) return OB_OK;
  if ((st = check_ls(ctx, ls, true))) return st;
  OB_CHECK_PTR(ctx, m, 16, "m");
  OB_CHECK_PTR(ctx, v, 16, "v");
  OB_CHECK_PTR(ctx, v_fresh, 16, "v_fresh");
  if (warmup_steps < 1)
    return fail(ctx, OB_ERR_INVALID, "warmup_steps = %d must be >= 1", warmup_steps);
  e = cudaMemcpyAsync(v_fresh, v, G.n_pad * sizeof(float), cudaMemcpyDeviceToDevice, s);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "begin_compression: v_fresh = v");
  ob::WarmupArgs a{};
  a.geo = G;
  a.ws = ctx->ws;
  a.m = const_cast<float*>(m);
  a.ls = *ls;
  a.warmup_steps = warmup_steps;
  return launched(ctx, ob::launch_lamb_begin(a, ctx->sms, s), "begin_compression");
}

ob_status ob_compress(ob_ctx* ctx, const void* const* grads, const float* m, float* const* err,
                      uint32_t* bits, float* scales, const ob_layer_state* ls,
                      ob_stream_t stream) {
  OB_TRACE();
  ob_status st = ready(ctx);
  if (st) return st;
  if ((st = check_grads(ctx, grads)) || (st = check_errs(ctx, err))) return st;
  OB_CHECK_PTR(ctx, m, 16, "m");
  OB_CHECK_PTR(ctx, bits, 16, "bits");
  OB_CHECK_PTR(ctx, scales, 4, "scales");
  if (ls && (st = check_ls(ctx, ls, false))) return st;
  ob::CompressArgs a{};
  a.geo = ctx->geo;
  a.ws = ctx->ws;
  a.nw = ctx->geo.W;
  for (int w = 0; w < ctx->cfg.W; ++w) {
    a.g[w] = grads[w];
    a.e[w] = err[w];
  }
  a.m = m;
  a.bits = bits;
  a.scales = scales;
  if (ls) {
    a.s = ls->s;
    a.c_prev = ls->c_prev;
    a.c_prev2 = ls->c_prev2;
  }
  a.ratio_ef = (ctx->cfg.flags & OB_FLAG_NO_RATIO_EF) ? 0 : 1;
  a.b1 = ctx->cfg.b1;
  a.ob1 = 1.0f - ctx->cfg.b1;
  a.clip = ctx->cfg.clip_value;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if ((st = launched(ctx,
                     ob::launch_compress(a, ctx->cfg.grad_dtype == OB_GRAD_BF16, ls != nullptr,
                                         ctx->sms, s),
                     "compress")))
    return st;
  return launched(ctx,
                  ob::launch_finalize_scales(ctx->geo, ctx->ws.wpart, ctx->geo.W, scales,
                                             ctx->sms, s),
                  "compress: chunk scales");
}

// Two device ranges [a, a+na) and [b, b+nb) share a byte.
static bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

static ob_status server_reduce(ob_ctx* ctx, const uint32_t* bits, const float* scales,
                               float* err_s, const uint32_t* sbits_old, const float* sscales_old,
                               uint32_t* sbits, float* sscales, const ob_layer_state* ls,
                               ob_stream_t stream) {
  ob_status st = ready(ctx);
  if (st) return st;
  OB_CHECK_PTR(ctx, bits, 16, "bits");
  OB_CHECK_PTR(ctx, scales, 4, "scales");
  OB_CHECK_PTR(ctx, err_s, 16, "err_s");
  OB_CHECK_PTR(ctx, sbits_old, 16, "sbits_old");
  OB_CHECK_PTR(ctx, sscales_old, 4, "sscales_old");
  OB_CHECK_PTR(ctx, sbits, 16, "sbits");
  OB_CHECK_PTR(ctx, sscales, 4, "sscales");
  const size_t wb = (size_t)ctx->geo.words * sizeof(uint32_t), cb = (size_t)ctx->geo.nc * 4;
  if ((sbits_old != sbits && overlap(sbits_old, wb, sbits, wb)) ||
      (sscales_old != sscales && overlap(sscales_old, cb, sscales, cb)))
    return fail(ctx, OB_ERR_INVALID, "old and new server buffers overlap without being equal");
  if (ls && (st = check_ls(ctx, ls, false))) return st;
  ob::ServerArgs a{};
  a.geo = ctx->geo;
  a.ws = ctx->ws;
  a.T0 = 0;
  a.T1 = ctx->geo.n_tiles;
  a.bits_stride = ctx->geo.words;
  a.sc_stride = ctx->geo.nc;
  a.bits = bits;
  a.scales = scales;
  a.e_s = err_s;
  a.sbits = sbits;
  a.sscales = sscales;
  a.sbits_old = sbits_old;
  a.sscales_old = sscales_old;
  if (ls) {
    a.c_prev = ls->c_prev;
    a.c_prev2 = ls->c_prev2;
  }
  a.ratio_ef = (ctx->cfg.flags & OB_FLAG_NO_RATIO_EF) ? 0 : 1;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if ((st = launched(ctx, ob::launch_server(a, ls != nullptr, ctx->sms, s), "server_reduce")))
    return st;
  return launched(ctx, ob::launch_finalize_scales(ctx->geo, ctx->ws.spart, 1, sscales, ctx->sms, s),
                  "server_reduce: chunk scales");
}

ob_status ob_server_reduce(ob_ctx* ctx, const uint32_t* bits, const float* scales, float* err_s,
                           uint32_t* sbits, float* sscales, const ob_layer_state* ls,
                           ob_stream_t stream) {
  OB_TRACE();
  return server_reduce(ctx, bits, scales, err_s, sbits, sscales, sbits, sscales, ls, stream);
}

ob_status ob_server_reduce_db(ob_ctx* ctx, const uint32_t* bits, const float* scales,
                              float* err_s, const uint32_t* sbits_old, const float* sscales_old,
                              uint32_t* sbits, float* sscales, const ob_layer_state* ls,
                              ob_stream_t stream) {
  OB_TRACE();
  return server_reduce(ctx, bits, scales, err_s, sbits_old, sscales_old, sbits, sscales, ls,
                       stream);
}

static void fill_update(const ob_ctx* ctx, ob::UpdateArgs& a) {
  const ob_config& c = ctx->cfg;
  a.geo = ctx->geo;
  a.ws = ctx->ws;
  a.b1 = c.b1;
  a.ob1 = 1.0f - c.b1;
  a.b2 = c.b2;
  a.ob2 = 1.0f - c.b2;
  a.eps = c.eps;
  a.lr = c.lr;
  a.hp.r_thr = c.r_thr;
  a.hp.r_min = c.r_min;
  a.hp.r_max = c.r_max;
  a.hp.c_min = c.c_min;
  a.hp.c_max = c.c_max;
  a.hp.ratio_ef = (c.flags & OB_FLAG_NO_RATIO_EF) ? 0 : 1;
  a.hp.frozen = (c.flags & OB_FLAG_FROZEN_C) ? 1 : 0;
}

ob_status ob_decompress(ob_ctx* ctx, const uint32_t* sbits, const float* sscales,
                        const ob_layer_state* ls, float* out, ob_stream_t stream) {
  OB_TRACE();
  ob_status st = ready(ctx);
  if (st) return st;
  OB_CHECK_PTR(ctx, sbits, 16, "sbits");
  OB_CHECK_PTR(ctx, sscales, 4, "sscales");
  OB_CHECK_PTR(ctx, out, 16, "out");
  if (ls) OB_CHECK_PTR(ctx, ls->s, 4, "ls.s");
  ob::UpdateArgs a{};
  fill_update(ctx, a);
  a.sbits = sbits;
  a.sscales = sscales;
  a.out = out;
  if (ls) a.ls = *ls;
  return launched(ctx,
                  ob::launch_decompress(a, ls != nullptr, ctx->sms,
                                        reinterpret_cast<cudaStream_t>(stream)),
                  "decompress");
}

ob_status ob_adam_step(ob_ctx* ctx, const uint32_t* sbits, const float* sscales,
                       const float* v_frozen, float* m, float* p, ob_stream_t stream) {
  OB_TRACE();
  ob_status st = ready(ctx);
  if (st) return st;
  OB_CHECK_PTR(ctx, sbits, 16, "sbits");
  OB_CHECK_PTR(ctx, sscales, 4, "sscales");
  OB_CHECK_PTR(ctx, v_frozen, 16, "v_frozen");
  if (m && !aligned(m, 16)) return fail(ctx, OB_ERR_ALIGN, "m is not 16-byte aligned");
  OB_CHECK_PTR(ctx, p, 16, "p");
  ob::UpdateArgs a{};
  fill_update(ctx, a);
  a.sbits = sbits;
  a.sscales = sscales;
  a.v_frozen = v_frozen;
  a.m = m;  // may be null: the momentum stays in its sign form
  a.p = p;
  return launched(ctx,
                  ob::launch_adam_update(a, ctx->sms, reinterpret_cast<cudaStream_t>(stream)),
                  "adam_step");
}

// m != NULL: dense momentum (read as m_{t-1}, written as m_t); m == NULL:
// m_{t-1} from (sbits_prev, sscales_prev) and m_t not written.
static ob_status lamb_step(ob_ctx* ctx, const uint32_t* sbits_prev, const float* sscales_prev,
                           const uint32_t* sbits, const float* sscales, const float* v_frozen,
                           float* v_fresh, float* m, float* p, const ob_layer_state* ls,
                           ob_stream_t stream) {
  ob_status st = ready(ctx);
  if (st) return st;
  OB_CHECK_PTR(ctx, sbits, 16, "sbits");
  OB_CHECK_PTR(ctx, sscales, 4, "sscales");
  OB_CHECK_PTR(ctx, v_frozen, 16, "v_frozen");
  OB_CHECK_PTR(ctx, v_fresh, 16, "v_fresh");
  if (m) {
    OB_CHECK_PTR(ctx, m, 16, "m");
  } else {
    OB_CHECK_PTR(ctx, sbits_prev, 16, "sbits_prev");
    OB_CHECK_PTR(ctx, sscales_prev, 4, "sscales_prev");
    if (overlap(sbits_prev, (size_t)ctx->geo.words * 4, sbits, (size_t)ctx->geo.words * 4) ||
        overlap(sscales_prev, (size_t)ctx->geo.nc * 4, sscales, (size_t)ctx->geo.nc * 4))
      return fail(ctx, OB_ERR_INVALID, "the previous and current server buffers must be disjoint");
  }
  OB_CHECK_PTR(ctx, p, 16, "p");
  if ((st = check_ls(ctx, ls, false))) return st;
  ob::UpdateArgs a{};
  fill_update(ctx, a);
  a.sbits = sbits;
  a.sscales = sscales;
  a.sbits_prev = sbits_prev;
  a.sscales_prev = sscales_prev;
  a.v_frozen = v_frozen;
  a.v_fresh = v_fresh;
  a.m = m;
  a.p = p;
  a.ls = *ls;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if ((st = launched(ctx, ob::launch_lamb_pass_a(a, ctx->sms, s), "lamb_step pass A"))) return st;
  return launched(ctx, ob::launch_lamb_pass_b(a, ctx->sms, s), "lamb_step pass B");
}

ob_status ob_lamb_step(ob_ctx* ctx, const uint32_t* sbits, const float* sscales,
                       const float* v_frozen, float* v_fresh, float* m, float* p,
                       const ob_layer_state* ls, ob_stream_t stream) {
  OB_TRACE();
  ob_status st = ready(ctx);
  if (st) return st;
  OB_CHECK_PTR(ctx, m, 16, "m");
  return lamb_step(ctx, nullptr, nullptr, sbits, sscales, v_frozen, v_fresh, m, p, ls, stream);
}

ob_status ob_lamb_step_signm(ob_ctx* ctx, const uint32_t* sbits_prev, const float* sscales_prev,
                             const uint32_t* sbits, const float* sscales, const float* v_frozen,
                             float* v_fresh, float* p, const ob_layer_state* ls,
                             ob_stream_t stream) {
  OB_TRACE();
  return lamb_step(ctx, sbits_prev, sscales_prev, sbits, sscales, v_frozen, v_fresh, nullptr, p,
                   ls, stream);
}

ob_status ob_compress_signm_ls(ob_ctx* ctx, const void* const* grads, const uint32_t* sbits,
                               const float* sscales, float* const* err, uint32_t* bits,
                               float* scales, const ob_layer_state* ls, ob_stream_t stream) {
  OB_TRACE();
  ob_status st = ready(ctx);
  if (st) return st;
  if ((st = check_grads(ctx, grads)) || (st = check_errs(ctx, err))) return st;
  OB_CHECK_PTR(ctx, sbits, 16, "sbits");
  OB_CHECK_PTR(ctx, sscales, 4, "sscales");
  OB_CHECK_PTR(ctx, bits, 16, "bits");
  OB_CHECK_PTR(ctx, scales, 4, "scales");
  if (ls && (st = check_ls(ctx, ls, false))) return st;
  ob::CompressArgs a{};
  a.geo = ctx->geo;
  a.ws = ctx->ws;
  a.nw = ctx->geo.W;
  for (int w = 0; w < ctx->cfg.W; ++w) {
    a.g[w] = grads[w];
    a.e[w] = err[w];
  }
  a.msbits = sbits;
  a.msscales = sscales;
  a.bits = bits;
  a.scales = scales;
  if (ls) {
    a.s = ls->s;
    a.c_prev = ls->c_prev;
    a.c_prev2 = ls->c_prev2;
  }
  a.ratio_ef = (ctx->cfg.flags & OB_FLAG_NO_RATIO_EF) ? 0 : 1;
  a.b1 = ctx->cfg.b1;
  a.ob1 = 1.0f - ctx->cfg.b1;
  a.clip = ctx->cfg.clip_value;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if ((st = launched(ctx,
                     ob::launch_compress_signm(a, ctx->cfg.grad_dtype == OB_GRAD_BF16,
                                               ls != nullptr, ctx->sms, s),
                     "compress_signm")))
    return st;
  return launched(ctx,
                  ob::launch_finalize_scales(ctx->geo, ctx->ws.wpart, ctx->geo.W, scales,
                                             ctx->sms, s),
                  "compress_signm: chunk scales");
}

ob_status ob_compress_signm(ob_ctx* ctx, const void* const* grads, const uint32_t* sbits,
                            const float* sscales, float* const* err, uint32_t* bits,
                            float* scales, ob_stream_t stream) {
  OB_TRACE();
  return ob_compress_signm_ls(ctx, grads, sbits, sscales, err, bits, scales, nullptr, stream);
}

ob_status ob_step(ob_ctx* ctx, const void* const* grads, float* m, float* const* err,
                  uint32_t* bits, float* scales, float* err_s, uint32_t* sbits, float* sscales,
                  const float* v_frozen, float* v_fresh, float* p, const ob_layer_state* ls,
                  ob_stream_t stream) {
  OB_TRACE();
  ob_status st;
  if (!m && !ls) {
    // 1-bit Adam with the momentum held in its sign form
    if ((st = ob_compress_signm(ctx, grads, sbits, sscales, err, bits, scales, stream))) return st;
    if ((st = ob_server_reduce(ctx, bits, scales, err_s, sbits, sscales, nullptr, stream)))
      return st;
    return ob_adam_step(ctx, sbits, sscales, v_frozen, nullptr, p, stream);
  }
  st = ob_compress(ctx, grads, m, err, bits, scales, ls, stream);
  if (st) return st;
  if ((st = ob_server_reduce(ctx, bits, scales, err_s, sbits, sscales, ls, stream))) return st;
  if (!ls) return ob_adam_step(ctx, sbits, sscales, v_frozen, m, p, stream);
  return ob_lamb_step(ctx, sbits, sscales, v_frozen, v_fresh, m, p, ls, stream);
}

ob_status ob_step_db(ob_ctx* ctx, const void* const* grads, float* const* err, uint32_t* bits,
                     float* scales, float* err_s, const uint32_t* sbits_prev,
                     const float* sscales_prev, uint32_t* sbits, float* sscales,
                     const float* v_frozen, float* v_fresh, float* p, const ob_layer_state* ls,
                     ob_stream_t stream) {
  OB_TRACE();
  ob_status st;
  if ((st = ob_compress_signm_ls(ctx, grads, sbits_prev, sscales_prev, err, bits, scales, ls,
                                 stream)))
    return st;
  if ((st = ob_server_reduce_db(ctx, bits, scales, err_s, sbits_prev, sscales_prev, sbits,
                                sscales, ls, stream)))
    return st;
  if (!ls) return ob_adam_step(ctx, sbits, sscales, v_frozen, nullptr, p, stream);
  return ob_lamb_step_signm(ctx, sbits_prev, sscales_prev, sbits, sscales, v_frozen, v_fresh, p,
                            ls, stream);
}

ob_status ob_materialize_errors(ob_ctx* ctx, float* const* err, const uint32_t* bits,
                                float* scales, float* err_s, const uint32_t* sbits,
                                float* sscales, ob_stream_t stream) {
  OB_TRACE();
  ob_status st = ready(ctx);
  if (st) return st;
  if ((st = check_errs(ctx, err))) return st;
  OB_CHECK_PTR(ctx, bits, 16, "bits");
  OB_CHECK_PTR(ctx, scales, 4, "scales");
  OB_CHECK_PTR(ctx, err_s, 16, "err_s");
  OB_CHECK_PTR(ctx, sbits, 16, "sbits");
  OB_CHECK_PTR(ctx, sscales, 4, "sscales");
  const Geo& G = ctx->geo;
  ob::MaterializeArgs a{};
  a.geo = G;
  a.nw = G.W;
  a.T1 = G.n_tiles;
  for (uint32_t w = 0; w < G.W; ++w) a.e[w] = err[w];
  a.bits = bits;
  a.scales = scales;
  a.e_s = err_s;
  a.sbits = sbits;
  a.sscales = sscales;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if ((st = launched(ctx, ob::launch_materialize(a, ctx->sms, s), "materialize"))) return st;
  cudaError_t e = cudaMemsetAsync(scales, 0, (size_t)G.W * G.nc * sizeof(float), s);
  if (e == cudaSuccess) e = cudaMemsetAsync(sscales, 0, (size_t)G.nc * sizeof(float), s);
  return launched(ctx, e, "materialize: clearing the scales");
}

ob_status ob_reset_errors(ob_ctx* ctx, float* const* err, const uint32_t* bits,
                          const float* scales, float* err_s, const uint32_t* sbits,
                          const float* sscales, ob_stream_t stream) {
  OB_TRACE();
  ob_status st = ready(ctx);
  if (st) return st;
  if ((st = check_errs(ctx, err))) return st;
  OB_CHECK_PTR(ctx, bits, 16, "bits");
  OB_CHECK_PTR(ctx, scales, 4, "scales");
  OB_CHECK_PTR(ctx, err_s, 16, "err_s");
  OB_CHECK_PTR(ctx, sbits, 16, "sbits");
  OB_CHECK_PTR(ctx, sscales, 4, "sscales");
  const Geo& G = ctx->geo;
  ob::MaterializeArgs a{};
  a.geo = G;
  a.nw = G.W;
  a.T1 = G.n_tiles;
  for (uint32_t w = 0; w < G.W; ++w) a.e[w] = err[w];
  a.bits = bits;
  a.scales = scales;
  a.e_s = err_s;
  a.sbits = sbits;
  a.sscales = sscales;
  return launched(ctx,
                  ob::launch_reset_errors(a, ctx->sms, reinterpret_cast<cudaStream_t>(stream)),
                  "reset_errors");
}

ob_status ob_error_norm(ob_ctx* ctx, const float* const* err, const uint32_t* bits,
                        const float* scales, const float* err_s, const uint32_t* sbits,
                        const float* sscales, float* out, ob_stream_t stream) {
  OB_TRACE();
  ob_status st = ready(ctx);
  if (st) return st;
  if ((st = check_errs(ctx, const_cast<float* const*>(err)))) return st;
  OB_CHECK_PTR(ctx, bits, 16, "bits");
  OB_CHECK_PTR(ctx, scales, 4, "scales");
  OB_CHECK_PTR(ctx, err_s, 16, "err_s");
  OB_CHECK_PTR(ctx, sbits, 16, "sbits");
  OB_CHECK_PTR(ctx, sscales, 4, "sscales");
  OB_CHECK_PTR(ctx, out, 4, "out");
  const Geo& G = ctx->geo;
  ob::MaterializeArgs a{};
  a.geo = G;
  a.nw = G.W;
  a.T1 = G.n_tiles;
  for (uint32_t w = 0; w < G.W; ++w) a.e[w] = const_cast<float*>(err[w]);
  a.bits = bits;
  a.scales = scales;
  a.e_s = const_cast<float*>(err_s);
  a.sbits = sbits;
  a.sscales = sscales;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if ((st = launched(ctx, ob::launch_error_norm(a, ctx->ws, ctx->sms, s), "error_norm")))
    return st;
  if ((st = launched(ctx, ob::launch_finalize_sums(G, ctx->ws.wpart, G.W, out, ctx->sms, s),
                     "error_norm: worker sums")))
    return st;
  return launched(ctx,
                  ob::launch_finalize_sums(G, ctx->ws.spart, 1, out + (size_t)G.W * G.nc,
                                           ctx->sms, s),
                  "error_norm: server sums");
}

ob_status ob_device_error(ob_ctx* ctx, unsigned* code, ob_stream_t stream) {
  OB_TRACE();
  ob_status st = ready(ctx);
  if (st) return st;
  if (!code) return fail(ctx, OB_ERR_INVALID, "code is NULL");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  unsigned v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, ctx->ws.err, sizeof v, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(ctx->ws.err, 0, sizeof v, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "device_error");
  *code = v;
  return OB_OK;
}

ob_status ob_quant_int8(const float* g, size_t n, int8_t* q, float* block_scales, uint64_t seed,
                        uint64_t step, float* deq, ob_stream_t stream) {
  OB_TRACE();
  if (n < 1 || n >= (1ull << 34))
    return fail(nullptr, OB_ERR_INVALID, "n = %zu must be in [1, 2^34)", n);
  OB_CHECK_PTR(nullptr, g, 16, "g");
  OB_CHECK_PTR(nullptr, q, 4, "q");
  OB_CHECK_PTR(nullptr, block_scales, 4, "block_scales");
  if (deq && !aligned(deq, 16)) return fail(nullptr, OB_ERR_ALIGN, "deq is not 16-byte aligned");
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(nullptr, e, "device query");
  e = ob::launch_quant_int8(g, n, q, block_scales, seed, step, deq, sms,
                            reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(nullptr, e, "quant_int8");
  return OB_OK;
}

ob_status ob_quant_int8_ef(const float* g, float* e, size_t n, int8_t* q, float* block_scales,
                           uint64_t seed, uint64_t step, float* deq, float* block_err2,
                           ob_stream_t stream) {
  OB_TRACE();
  if (n < 1 || n >= (1ull << 34))
    return fail(nullptr, OB_ERR_INVALID, "n = %zu must be in [1, 2^34)", n);
  OB_CHECK_PTR(nullptr, g, 16, "g");
  OB_CHECK_PTR(nullptr, e, 16, "e");
  OB_CHECK_PTR(nullptr, q, 4, "q");
  OB_CHECK_PTR(nullptr, block_scales, 4, "block_scales");
  if (deq && !aligned(deq, 16)) return fail(nullptr, OB_ERR_ALIGN, "deq is not 16-byte aligned");
  if (block_err2 && !aligned(block_err2, 4))
    return fail(nullptr, OB_ERR_ALIGN, "block_err2 is not 4-byte aligned");
  int dev = 0, sms = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err == cudaSuccess) err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return cuda_fail(nullptr, err, "device query");
  err = ob::launch_quant_int8_ef(g, e, n, q, block_scales, seed, step, deq, block_err2, sms,
                                 reinterpret_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(nullptr, err, "quant_int8_ef");
  return OB_OK;
}

}  // extern "C"
