// Internal declarations shared by the libob translation units: the layout
// ("geometry") handed to every kernel, the kernel argument blocks, the
// device helpers for tile decoding, the fixed-order tile reduction and sign
// packing, and the host-side launchers.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include "ob.h"

namespace ob {

constexpr int kThreads = 256;      // one CTA = the 256 lanes of a tile
constexpr uint32_t kTile = 4096;   // elements per tile
constexpr unsigned kFull = 0xffffffffu;

// Layout of the fused buffer, as the kernels see it.
struct Geo {
  uint64_t n;        // real elements
  uint64_t P;        // partition size (multiple of 32)
  uint64_t C;        // chunk size, <= P, multiple of 32
  uint64_t Cl;       // length of the last chunk of a partition
  uint64_t n_pad;    // W * P
  uint64_t words;    // row stride of the sign words: n_pad/32 rounded up to 4
  uint32_t W;        // workers
  uint32_t cpp;      // chunks per partition
  uint32_t tpc;      // tiles in a full chunk (also the stride of partials)
  uint32_t tpl;      // tiles in the last chunk of a partition
  uint32_t tpp;      // tiles per partition
  uint32_t nc;       // chunks in total, W * cpp
  uint32_t n_tiles;  // tiles in total, W * tpp
  uint32_t L;        // layers (>= 1)
  uint32_t n_ltiles; // tiles counted per layer (from each layer's start)
};

// One tile of 4096 (or fewer) elements inside one chunk.
struct Tile {
  uint64_t start;   // first element
  uint64_t cstart;  // first element of its chunk
  uint64_t real;    // real (non-padding) elements of its chunk
  uint32_t len;     // elements in the tile, multiple of 32, <= 4096
  uint32_t g;       // chunk id
  uint32_t t;       // index of the tile inside its chunk
  uint32_t ntc;     // tiles in its chunk
};

__device__ __forceinline__ Tile decode_tile(const Geo& G, uint32_t T) {
  Tile r;
  uint32_t j = T / G.tpp;
  uint32_t rem = T - j * G.tpp;
  uint32_t kc = rem / G.tpc;  // the last chunk has tpl <= tpc tiles
  r.t = rem - kc * G.tpc;
  bool last = (kc == G.cpp - 1);
  uint64_t clen = last ? G.Cl : G.C;
  r.ntc = last ? G.tpl : G.tpc;
  r.g = j * G.cpp + kc;
  r.cstart = (uint64_t)j * G.P + (uint64_t)kc * G.C;
  r.start = r.cstart + (uint64_t)r.t * kTile;
  uint64_t left = clen - (uint64_t)r.t * kTile;
  r.len = (uint32_t)(left < kTile ? left : kTile);
  r.real = G.n > r.cstart ? (G.n - r.cstart < clen ? G.n - r.cstart : clen) : 0;
  return r;
}

// Workspace regions (byte offsets from the workspace base).
struct Workspace {
  float* wpart;          // [W][nc][tpc] worker tile totals
  float* spart;          // [nc][tpc] server tile totals
  uint32_t* tile_layer;  // [n_tiles] layer of each tile's first element
  uint64_t* layer_off;   // [L+1]
  uint32_t* ltile_pref;  // [L+1] prefix count of per-layer tiles
  float* lpart;          // [2][n_ltiles] per-layer tile totals
  unsigned* Rbits;       // [L] LAMB max ratio, as float bit patterns
  float* rms;            // [L] begin: momentum RMS per layer
  unsigned* gcnt;        // [4] whole-grid arrival counters (LAMB pass A)
  unsigned* err;         // [1] first device-side error code (0 = none)
};

// LAMB per-layer parameters handed to kernels.
struct LambHP {
  float r_thr, r_min, r_max, c_min, c_max;
  int ratio_ef;  // 1: rho = c_{t-2}/c_{t-1}; 0: rho = 1
  int frozen;    // 1: r = 1, c = c_avg
};

// ---------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------

// Warp butterfly: every lane ends with the same value; lane l adds the
// value of lane l^o for o = 16, 8, 4, 2, 1.
__device__ __forceinline__ float warp_butterfly_sum(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

// Pairwise tree over the 8 warp totals of a tile.
__device__ __forceinline__ float tree8(const float* w) {
  float s01 = __fadd_rn(w[0], w[1]), s23 = __fadd_rn(w[2], w[3]);
  float s45 = __fadd_rn(w[4], w[5]), s67 = __fadd_rn(w[6], w[7]);
  return __fadd_rn(__fadd_rn(s01, s23), __fadd_rn(s45, s67));
}

// OR of a 4-bit group over the 8 lanes that share one 32-bit word: lane l
// holds bits 4*(l%8)..4*(l%8)+3 of word l/8 of its warp's 128 elements.
__device__ __forceinline__ uint32_t pack_word(uint32_t nibble, int lane) {
  uint32_t w = nibble << (4 * (lane & 7));
  w |= __shfl_xor_sync(kFull, w, 1);
  w |= __shfl_xor_sync(kFull, w, 2);
  w |= __shfl_xor_sync(kFull, w, 4);
  return w;
}

// Sequential sum of `cnt` tile totals (from 0, in order), done by one warp:
// every lane returns the same value.  Each batch of 256 totals is loaded at
// once (8 per lane) and handed to the adding chain by shuffles, so only the
// additions are serialised: a full batch through unrolled shuffles, the
// last partial one through as many shuffles as it has totals (a one-tile
// chunk costs one).
__device__ __forceinline__ float ordered_sum(const float* part, uint32_t cnt, int lane) {
  float acc = 0.0f;
  for (uint32_t t0 = 0; t0 < cnt; t0 += 256) {
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t t = t0 + 32u * j + lane;
      v[j] = t < cnt ? __ldcg(part + t) : 0.0f;
    }
    const uint32_t rem = cnt - t0;  // the same in every lane
    if (rem >= 256) {
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int s = 0; s < 32; ++s) acc = __fadd_rn(acc, __shfl_sync(kFull, v[j], s));
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (32u * j >= rem) break;
        const uint32_t lim = rem - 32u * j < 32u ? rem - 32u * j : 32u;
        for (uint32_t s = 0; s < lim; ++s) acc = __fadd_rn(acc, __shfl_sync(kFull, v[j], s));
      }
    }
  }
  return acc;
}

// z / W for the server averages.  When W is a power of two, 1/W is exact
// and z * (1/W) is the same correctly rounded number as z / W (both round
// the same real value), so a multiply replaces the division; inv_w is
// 1/W then and 0 otherwise.
// +s if bit b of w is set, else -s: the sign bit of s flipped when the bit
// is clear -- the same value as the select, for -0 and NaN too, in two
// integer instructions.
__device__ __forceinline__ float signed_by_bit(float s, uint32_t w, int b) {
  return __uint_as_float(__float_as_uint(s) ^ (~(w << (31 - b)) & 0x80000000u));
}

__device__ __forceinline__ float div_by_workers(float z, float fW, float inv_w) {
  return inv_w != 0.0f ? __fmul_rn(z, inv_w) : __fdiv_rn(z, fW);
}

__host__ __device__ inline float inv_workers(uint32_t W) {
  return (W & (W - 1)) == 0 ? 1.0f / (float)W : 0.0f;
}

__device__ __forceinline__ float mean_of(float sum, uint64_t count) {
  return count ? __fdiv_rn(sum, __ull2float_rn(count)) : 0.0f;
}

// Two fp32 values in one 64-bit register pair, and the paired IEEE addition
// of sm_100-class GPUs (PTX add.rn.f32x2): each half is rounded on its own,
// to nearest even, with subnormals kept -- the result of __fadd_rn on that
// half -- in one instruction for both.
__device__ __forceinline__ unsigned long long f2_make(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_split(unsigned long long a, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(a));
}
__device__ __forceinline__ unsigned long long f2_add(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

__device__ __forceinline__ float fmax_plain(float a, float b) { return a > b ? a : b; }
__device__ __forceinline__ float fmin_plain(float a, float b) { return a < b ? a : b; }

__device__ __forceinline__ float bf16_to_f32(uint16_t h) {
  return __uint_as_float(((uint32_t)h) << 16);
}

// Loads 4 gradient values starting at element k (16-byte / 8-byte aligned).
template <bool BF16>
__device__ __forceinline__ float4 load_grad4(const void* g, uint64_t k) {
  if constexpr (BF16) {
    uint2 u = __ldcs(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(g) + k));
    float4 r;
    r.x = __uint_as_float(u.x << 16);
    r.y = __uint_as_float(u.x & 0xffff0000u);
    r.z = __uint_as_float(u.y << 16);
    r.w = __uint_as_float(u.y & 0xffff0000u);
    return r;
  } else {
    return __ldcs(reinterpret_cast<const float4*>(static_cast<const float*>(g) + k));
  }
}

__device__ __forceinline__ float& f4at(float4& v, int c) {
  return c == 0 ? v.x : c == 1 ? v.y : c == 2 ? v.z : v.w;
}
__device__ __forceinline__ float f4get(const float4& v, int c) {
  return c == 0 ? v.x : c == 1 ? v.y : c == 2 ? v.z : v.w;
}

// Layer tracking: advances `l` until element k lies in [off[l], off[l+1]).
__device__ __forceinline__ bool advance_layer(const uint64_t* off, uint32_t L,
                                              uint64_t k, uint32_t& l,
                                              uint64_t& lend) {
  bool moved = false;
  while (k >= lend && l + 1 < L) {
    ++l;
    lend = __ldg(off + l + 1);
    moved = true;
  }
  return moved;
}

// ---------------------------------------------------------------------------
// Kernel argument blocks
// ---------------------------------------------------------------------------

struct CompressArgs {
  Geo geo;
  Workspace ws;
  uint32_t nw;             // workers compressed by this call: geo.W, or 1 for one
                           // rank's own worker (its buffers are g[0], e[0], row 0)
  const void* g[OB_MAX_WORKERS];
  float* e[OB_MAX_WORKERS];
  const float* m;          // dense momentum, or null: then m = msscale*sign(msbits)
  const uint32_t* msbits;  // momentum in sign form (the previous server step)
  const float* msscales;
  uint32_t* bits;
  float* scales;
  const float* s;        // LAMB sigma, or null
  const float* c_prev;   // LAMB c_{t-1}
  const float* c_prev2;  // LAMB c_{t-2}
  int ratio_ef;
  float b1, ob1;
  float clip;  // > 0: compensated values limited to [-clip, clip]
};

struct ServerArgs {
  Geo geo;
  Workspace ws;
  // The tiles [T0, T1) this call reduces: every tile, or one partition's
  // (one rank's server).  Index 0 of e_s, sbits and sbits_old is element
  // `base`, index 0 of sscales and sscales_old is chunk g0; the workers'
  // rows of bits are bits_stride words apart, those of scales sc_stride
  // floats apart.  The whole buffer: T0 = 0, T1 = n_tiles, base = g0 = 0,
  // strides words and nc.
  uint32_t T0, T1, g0, sc_stride;
  uint64_t base, bits_stride;
  const uint32_t* bits;
  const float* scales;
  float* e_s;
  uint32_t* sbits;
  float* sscales;
  const uint32_t* sbits_old;  // the previous server words and scales (the
  const float* sscales_old;   // deferred error's); == sbits/sscales unless double-buffered
  const float* c_prev;
  const float* c_prev2;
  int ratio_ef;
};

struct UpdateArgs {
  Geo geo;
  Workspace ws;
  const uint32_t* sbits;
  const float* sscales;
  const float* v_frozen;
  float* v_fresh;
  float* m;              // null: the momentum is held in sign form
  const uint32_t* sbits_prev;  // LAMB, sign form: the previous step's server words
  const float* sscales_prev;   // and scales (m_{t-1} = sscale*sign/sigma)
  float* p;
  float* out;            // decompress
  ob_layer_state ls;     // LAMB arrays (device pointers)
  LambHP hp;
  float b1, ob1, b2, ob2, eps, lr;
};

struct MaterializeArgs {
  Geo geo;
  float* e[OB_MAX_WORKERS];
  const uint32_t* bits;
  const float* scales;
  float* e_s;
  const uint32_t* sbits;
  const float* sscales;
  // k_materialize: workers 0..nw-1 (rows of bits and scales) and, if e_s is
  // set, the server, over the tiles [T0, T1); the server's element k is at
  // index k - base of e_s and sbits, its chunk g at g - g0 of sscales.  The
  // whole buffer: nw = W, T0 = 0, T1 = n_tiles, base = g0 = 0.
  uint32_t nw, T0, T1, g0;
  uint64_t base;
};

struct WarmupArgs {
  Geo geo;
  Workspace ws;
  const void* g[OB_MAX_WORKERS];
  float* m;
  float* v;
  float* p;
  ob_layer_state ls;
  float b1, ob1, b2, ob2, eps, lr, c_min, c_max;
  float fW, inv_w;  // W, and 1/W when W is a power of two (else 0)
  int warmup_steps;
};

// Layerwise mixed widths: the b-bit codec (blocks of 256, codes packed BITS
// to an element) and the FP16 codec.
struct QbCompressArgs {
  const void* g[OB_MAX_WORKERS];
  float* e[OB_MAX_WORKERS];
  const float* m;
  uint32_t* codes;     // [W][row_words]
  float* scales;       // [W][n_pad/256]
  uint64_t n, n_pad, row_words, seed, step;
  uint32_t W;
  float b1, clip;
};

struct QbServerArgs {
  const uint32_t* codes;
  const float* scales;
  float* e_s;
  uint32_t* scodes;
  float* sscales;
  uint64_t n, n_pad, row_words, seed, step;
  uint32_t W;
};

struct QbUpdateArgs {
  const uint32_t* scodes;
  const float* sscales;
  const float* v;
  float* m;
  float* p;
  uint64_t n, n_pad;
  float lr, eps;
};

struct F16Args {
  const void* g[OB_MAX_WORKERS];
  float* e[OB_MAX_WORKERS];
  float* m;            // read by the worker kernel, written by the update
  uint16_t* h;         // [W][n_pad] worker messages
  uint16_t* hs;        // [n_pad] server message
  float* e_s;
  const float* v;
  float* p;
  uint64_t n, n_pad;
  uint32_t W;
  int send;
  float b1, clip, lr, eps;
};

// ---------------------------------------------------------------------------
// Launchers.  Each sizes its grid to the CTAs that fit on the device at once
// (SM count x resident CTAs per SM, at most one CTA per tile) and returns
// the cudaError_t of its launch.
// ---------------------------------------------------------------------------

// One NVTX range, named after the C entry point, for the duration of each
// ob_* call, so that the library's calls show up by name on a profiler's
// timeline next to the caller's own work.  Without a tool attached an NVTX
// call costs one indirect call.
struct TraceRange {
  explicit TraceRange(const char* name) { nvtxRangePushA(name); }
  ~TraceRange() { nvtxRangePop(); }
  TraceRange(const TraceRange&) = delete;
  TraceRange& operator=(const TraceRange&) = delete;
};
#define OB_TRACE() ::ob::TraceRange ob_trace_range_(__func__)

// Views of a ctx (defined with the C entry points).
const Geo* ctx_geo(const ob_ctx* ctx);
const Workspace* ctx_ws(const ob_ctx* ctx);  // null before ob_set_workspace
int ctx_sms(const ob_ctx* ctx);
const ob_config* ctx_config(const ob_ctx* ctx);
ob_status ctx_fail(ob_ctx* ctx, ob_status st, const char* msg);

// Runs a setup call (e.g. a kernel's dynamic shared-memory limit, which
// is a per-device attribute) once on each device the process uses; one
// instance per call site.
struct PerDeviceOnce {
  std::atomic<uint64_t> done{0};  // bit d: done on device d (< 64)
  template <typename F>
  cudaError_t run(F f) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    e = f();
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
  }
};

template <typename K>
inline int grid_for(K kernel, int sms, uint64_t items, int threads = kThreads,
                    size_t smem = 0) {
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, threads, smem) != cudaSuccess ||
      occ < 1)
    occ = 1;
  uint64_t g = (uint64_t)sms * (uint64_t)occ;
  if (g > items) g = items;
  if (g < 1) g = 1;
  return (int)g;
}

cudaError_t launch_compress(const CompressArgs& a, bool bf16, bool lamb, int sms,
                            cudaStream_t s);
cudaError_t launch_compress_signm(const CompressArgs& a, bool bf16, bool lamb, int sms,
                                  cudaStream_t s);
cudaError_t launch_server(const ServerArgs& a, bool lamb, int sms, cudaStream_t s);
cudaError_t launch_finalize_scales(const Geo& G, const float* part, uint32_t rows,
                                   float* scales, int sms, cudaStream_t s);
cudaError_t launch_finalize_sums(const Geo& G, const float* part, uint32_t rows, float* sums,
                                 int sms, cudaStream_t s);
// The scales of chunks [g0, g0 + count) of `rows` rows into scales[row][count].
cudaError_t launch_finalize_scales_range(const Geo& G, const float* part, uint32_t rows,
                                         uint32_t g0, uint32_t count, float* scales, int sms,
                                         cudaStream_t s);
cudaError_t launch_error_norm(const MaterializeArgs& a, const Workspace& ws, int sms,
                              cudaStream_t s);
cudaError_t launch_adam_update(const UpdateArgs& a, int sms, cudaStream_t s);
cudaError_t launch_lamb_pass_a(const UpdateArgs& a, int sms, cudaStream_t s);
cudaError_t launch_lamb_pass_b(const UpdateArgs& a, int sms, cudaStream_t s);
cudaError_t launch_decompress(const UpdateArgs& a, bool layered, int sms,
                              cudaStream_t s);
cudaError_t launch_materialize(const MaterializeArgs& a, int sms, cudaStream_t s);
cudaError_t launch_reset_errors(const MaterializeArgs& a, int sms, cudaStream_t s);
cudaError_t launch_qb_compress(const QbCompressArgs& a, int bits, bool bf16, int sms,
                               cudaStream_t s);
cudaError_t launch_qb_server(const QbServerArgs& a, int bits, int sms, cudaStream_t s);
cudaError_t launch_qb_adam(const QbUpdateArgs& a, int bits, int sms, cudaStream_t s);
cudaError_t launch_f16_compress(const F16Args& a, bool bf16, int sms, cudaStream_t s);
cudaError_t launch_f16_server(const F16Args& a, int sms, cudaStream_t s);
cudaError_t launch_f16_adam(const F16Args& a, int sms, cudaStream_t s);
cudaError_t launch_warmup_adam(const WarmupArgs& a, bool bf16, int sms,
                               cudaStream_t s);
cudaError_t launch_warmup_lamb(const WarmupArgs& a, bool bf16, int sms,
                               cudaStream_t s);
cudaError_t launch_lamb_begin(const WarmupArgs& a, int sms, cudaStream_t s);
cudaError_t launch_quant_int8(const float* g, uint64_t n, int8_t* q, float* scales,
                              uint64_t seed, uint64_t step, float* deq, int sms,
                              cudaStream_t s);
cudaError_t launch_quant_int8_ef(const float* g, float* e, uint64_t n, int8_t* q, float* scales,
                                 uint64_t seed, uint64_t step, float* deq, float* err2, int sms,
                                 cudaStream_t s);

}  // namespace ob
