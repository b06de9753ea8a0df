// Oracle for the error-compensated 1-bit compressed optimizer step
// (1-bit Adam / 1-bit LAMB), the block-wise INT8 stochastic-rounding
// quantizer, and the layerwise mixed-width codecs (b-bit blocks, FP16).
//
// TEST INFRASTRUCTURE ONLY.  This file is a plain, slow, single-threaded
// restatement of the method, written to be checked by eye against the
// pages it follows.  Only tests/, __graft_entry__.smoke() and bench.py's
// CPU-baseline leg may load it.  It shares no code, header, table or helper
// with the CUDA library in momentum_compression_gb300/csrc/.
//
// Sources (cited by page title and section):
//   [BLOG]  lqnn.cn, "1bit Adam" practitioner write-up:
//           §2.1 error compensation (m/v recurrences; g' = g + e, q = sign(g'),
//           e = g' - q), §6 tuning config (warmup without quantization).
//   [TUT]   FreeGuideOnline, "梯度量化：将梯度从 FP32 压到 INT8 甚至 1-bit":
//           "FP32 → INT8 量化" (scale = max|g|/127, block-wise scales,
//           stochastic rounding), "1-bit 梯度量化" (scaled sign
//           mean(|g|)*sign(g), error feedback), and the GradientQuantizeINT8
//           example (floor + Bernoulli(frac), clamp to ±127).
//   [LAMB]  "1-bit LAMB (Error-Compensated LAMB-Preconditioned Large-Batch
//           Compressed Optimization)": ¶1 reconstructed g_t, fresh v_t, the
//           clipped infinity-norm ratio r_t and the frozen denominator;
//           ¶2 the fixed per-layer momentum scale and the fused 1-D buffer;
//           ¶3 step-ratio-scaled error feedback and the global-momentum
//           identity with the server error delta~; ¶4 the 3-phase
//           worker -> server -> worker compressed exchange.
//
// Arithmetic: IEEE binary32, every operation rounded on its own.  Build with
// -O2 -ffp-contract=off and without -ffast-math, so that no multiply-add is
// contracted and no subnormal is flushed.  Readings where the pages leave a
// step open are listed at each function.
//
// Layout (shared by every function; the pages fix none of it):
//   n real elements, W workers, alignment A, chunk C.
//   P = roundup(ceil(n/W), A); n_pad = W*P; server j owns [jP, (j+1)P).
//   Each partition is cut into chunks of C elements (the last may be short);
//   chunk g (global id) = partition g / cpp, chunk g % cpp within it,
//   cpp = ceil(P/C).  Elements k >= n are padding: they count nowhere,
//   their bit is 0 and their error is 0.
//   Bit rule: bit k%32 of word k/32 (LSB first) is 1 iff x[k] >= 0.0f, so
//   sign(+0) = sign(-0) = +1 and a NaN packs as -1.
//
// Parity pins: every function here is checked by tests/test_oracle_*.py
// against hand-computed values, closed forms, invariants, brute force or
// an independent library (curand's host Philox generator).

#include <cmath>
#include <cstddef>
#include <cstdint>
#include <cstring>
#include <vector>

extern "C" {

// ---------------------------------------------------------------------------
// Layout
// ---------------------------------------------------------------------------

struct orc_layout {
  uint64_t n, W, A, C;
  uint64_t P, n_pad, cpp, nc;
};

// Fills the derived sizes.  Returns 0, or -1 if the configuration is empty.
int orc_make_layout(uint64_t n, uint64_t W, uint64_t A, uint64_t C,
                    orc_layout* out) {
  if (W == 0 || A == 0 || C == 0 || out == nullptr) return -1;
  uint64_t per = (n + W - 1) / W;
  uint64_t P = (per + A - 1) / A * A;
  if (P == 0) P = A;  // n == 0 still has one aligned partition per worker
  uint64_t c = C < P ? C : P;
  out->n = n;
  out->W = W;
  out->A = A;
  out->C = c;
  out->P = P;
  out->n_pad = W * P;
  out->cpp = (P + c - 1) / c;
  out->nc = W * out->cpp;
  return 0;
}

static void chunk_range(const orc_layout* L, uint64_t g, uint64_t* start,
                        uint64_t* len, uint64_t* real) {
  uint64_t j = g / L->cpp, kc = g % L->cpp;
  uint64_t s = j * L->P + kc * L->C;
  uint64_t l = L->P - kc * L->C;
  if (l > L->C) l = L->C;
  uint64_t r = 0;
  if (L->n > s) r = (L->n - s < l) ? (L->n - s) : l;
  *start = s;
  *len = l;
  *real = r;
}

// ---------------------------------------------------------------------------
// Canonical reduction CR
// ---------------------------------------------------------------------------
// The order of every floating-point sum that decides a scale or a norm is
// fixed here, so that any implementation that follows it gets the same bits:
//   1. the segment is cut into tiles of 4096 elements from its own start;
//   2. inside a tile, lane p in [0,256) starts from 0 and adds, for i = 0..3
//      and then c = 0..3, element 1024*i + 4*p + c when present;
//   3. the 256 lanes are reduced in warps of 32 by a butterfly
//      (v[l] = v[l] + v[l ^ o], o = 16, 8, 4, 2, 1), and the 8 warp sums
//      pairwise: ((w0+w1)+(w2+w3)) + ((w4+w5)+(w6+w7));
//   4. the segment total is the sum of the tile totals, in tile order,
//      starting from 0.
// The pages only say "mean(abs(g))" (TUT, "1-bit 梯度量化") and "norm"; they
// fix no summation order.  `a` holds `count` present values; the segment
// may be longer, but absent elements (padding) are skipped, which is the
// same as ending it at `count`.

static float cr_tile(const float* a, uint64_t len) {
  float lane[256];
  for (int p = 0; p < 256; ++p) {
    float acc = 0.0f;
    for (int i = 0; i < 4; ++i)
      for (int c = 0; c < 4; ++c) {
        uint64_t idx = (uint64_t)(1024 * i + 4 * p + c);
        if (idx < len) acc = acc + a[idx];
      }
    lane[p] = acc;
  }
  float warp[8];
  for (int w = 0; w < 8; ++w) {
    float v[32];
    for (int l = 0; l < 32; ++l) v[l] = lane[32 * w + l];
    for (int o = 16; o >= 1; o >>= 1) {
      float nv[32];
      for (int l = 0; l < 32; ++l) nv[l] = v[l] + v[l ^ o];
      for (int l = 0; l < 32; ++l) v[l] = nv[l];
    }
    warp[w] = v[0];
  }
  float s01 = warp[0] + warp[1], s23 = warp[2] + warp[3];
  float s45 = warp[4] + warp[5], s67 = warp[6] + warp[7];
  float s0123 = s01 + s23, s4567 = s45 + s67;
  return s0123 + s4567;
}

float orc_cr_sum(const float* a, uint64_t count) {
  float total = 0.0f;
  for (uint64_t t = 0; t * 4096 < count; ++t) {
    uint64_t len = count - t * 4096;
    if (len > 4096) len = 4096;
    total = total + cr_tile(a + t * 4096, len);
  }
  return total;
}

// ---------------------------------------------------------------------------
// Per-layer lookups
// ---------------------------------------------------------------------------
// Layers are contiguous ranges of the fused 1-D buffer ([LAMB] ¶2):
// offsets[0] = 0 < offsets[1] < ... < offsets[nl] = n.  nl == 0 means one
// layer covering [0, n).

static uint64_t layer_of(const uint64_t* off, uint64_t nl, uint64_t k) {
  if (nl == 0) return 0;
  uint64_t lo = 0, hi = nl;  // invariant: off[lo] <= k < off[hi]
  while (hi - lo > 1) {
    uint64_t mid = (lo + hi) / 2;
    if (off[mid] <= k) lo = mid; else hi = mid;
  }
  return lo;
}

static float sgn_of_bit(const uint32_t* words, uint64_t k) {
  return ((words[k >> 5] >> (k & 31)) & 1u) ? 1.0f : -1.0f;
}

// ---------------------------------------------------------------------------
// Compressor C[x]: scaled sign with error feedback
// ---------------------------------------------------------------------------
// [TUT] "1-bit 梯度量化": q = mean(|x|) * sign(x); the error x - q is kept and
// added before the next compression ([BLOG] §2.1, e = g' - q; [TUT] error
// feedback).  The mean is taken per chunk (the fused buffer of [LAMB] ¶2 is
// cut into chunks); an all-padding chunk gets scale 0 (reading: the pages
// never divide by zero, and the value is never used for a real element).
//
// Worker side, for worker w (one call per worker):
//   m_w = b1*m + (1-b1)*g_w                        [BLOG] §2.1, momentum
//   x   = sigma_l*m_w + rho_l*e_w                  [LAMB] ¶2 (scale sigma_l
//         before compression) and ¶3 (step-ratio error feedback rho_l =
//         c_{t-2}/c_{t-1}); both are 1 for 1-bit Adam
//   scale(chunk) = CR(|x| over chunk) / realcount(chunk)
//   bit = x >= 0;  e_w' = x - scale*sign(x)
// `sigma`/`rho` are per-layer arrays or NULL (= 1).  e is updated in place.
// `x_out`, if not NULL, receives x (used by tests).
// clip > 0: the compensated value is limited to [-clip, clip] before it is
// compressed ([BLOG] §4.1 "梯度裁剪": compensated_grad.clamp_(-clip_value,
// clip_value), §6 clip_value 2.0); a NaN stays NaN.
// Chunk ranges.  Every output element of the compression, the server, the
// decompression and the updates depends only on its own chunk's inputs
// (LAMB's R is a running maximum), so the functions taking [g0, g1) do the
// same computation for chunks g0 <= g < g1 only, and the whole-buffer
// functions are these over [0, nc).  Disjoint ranges may run concurrently
// (each with its own R for pass A, merged by maximum) as long as no 32-bit
// word of bits/sbits holds elements of two of them, i.e. the range
// boundaries fall on multiples of 32 elements.
void orc_compress_worker_range(const orc_layout* L, const uint64_t* layer_off,
                               uint64_t nl, const float* sigma, const float* rho,
                               float b1, float clip, const float* g, const float* m,
                               float* e, uint32_t* bits, float* scales, float* x_out,
                               uint64_t g0, uint64_t g1) {
  const float ob1 = 1.0f - b1;
  std::vector<float> xs, ax;
  for (uint64_t g_id = g0; g_id < g1 && g_id < L->nc; ++g_id) {
    uint64_t start, len, real;
    chunk_range(L, g_id, &start, &len, &real);
    xs.assign(len, 0.0f);
    for (uint64_t q = 0; q < real; ++q) {
      uint64_t k = start + q;
      uint64_t l = layer_of(layer_off, nl, k);
      float s = sigma ? sigma[l] : 1.0f;
      float r = rho ? rho[l] : 1.0f;
      float mw = (b1 * m[k]) + (ob1 * g[k]);
      float xv = (s * mw) + (r * e[k]);
      if (clip > 0.0f) {
        if (xv > clip) xv = clip;
        if (xv < -clip) xv = -clip;
      }
      xs[q] = xv;
    }
    ax.assign(real, 0.0f);
    for (uint64_t q = 0; q < real; ++q) ax[q] = std::fabs(xs[q]);
    float sum = orc_cr_sum(ax.data(), real);
    float scale = real ? sum / (float)real : 0.0f;
    scales[g_id] = scale;
    for (uint64_t q = 0; q < len; ++q) {
      uint64_t k = start + q;
      bits[k >> 5] &= ~(1u << (k & 31));
      if (q < real) {
        float xv = xs[q];
        bool b = (xv >= 0.0f);
        if (b) bits[k >> 5] |= (1u << (k & 31));
        float sg = b ? 1.0f : -1.0f;
        e[k] = xv - (scale * sg);
      } else {
        e[k] = 0.0f;
      }
      if (x_out) x_out[k] = xs[q];
    }
  }
}

void orc_compress_worker_clip(const orc_layout* L, const uint64_t* layer_off,
                              uint64_t nl, const float* sigma, const float* rho,
                              float b1, float clip, const float* g, const float* m,
                              float* e, uint32_t* bits, float* scales, float* x_out) {
  for (uint64_t wd = 0; wd < L->n_pad / 32 + ((L->n_pad % 32) ? 1 : 0); ++wd)
    bits[wd] = 0u;
  orc_compress_worker_range(L, layer_off, nl, sigma, rho, b1, clip, g, m, e, bits, scales,
                            x_out, 0, L->nc);
}

void orc_compress_worker(const orc_layout* L, const uint64_t* layer_off,
                         uint64_t nl, const float* sigma, const float* rho,
                         float b1, const float* g, const float* m, float* e,
                         uint32_t* bits, float* scales, float* x_out) {
  orc_compress_worker_clip(L, layer_off, nl, sigma, rho, b1, 0.0f, g, m, e, bits,
                           scales, x_out);
}

// Server side, all partitions ([LAMB] ¶3-¶4: worker chunks travel to the
// server owning them, which averages, adds its own error delta~ and
// compresses again):
//   z_k = (sum over w = 0..W-1, in order, from 0, of scale_w(chunk)*sign_w(k)) / W
//   y   = rho_l*e_s + z
//   sscale(chunk) = CR(|y|) / realcount;  sbit = y >= 0;  e_s' = y - sscale*sign(y)
// bits: [W][n_pad/32] words; scales: [W][nc] (each worker's scale for every
// chunk of its full buffer).  Reading: the server uses the same chunking as
// the workers, and divides by W after the sum.
void orc_server_reduce_range(const orc_layout* L, const uint64_t* layer_off,
                             uint64_t nl, const float* rho, const uint32_t* bits,
                             const float* scales, float* e_s, uint32_t* sbits,
                             float* sscales, float* y_out, uint64_t g0, uint64_t g1) {
  const uint64_t words = L->n_pad / 32 + ((L->n_pad % 32) ? 1 : 0);
  const float fW = (float)L->W;
  std::vector<float> ys, ay;
  for (uint64_t g_id = g0; g_id < g1 && g_id < L->nc; ++g_id) {
    uint64_t start, len, real;
    chunk_range(L, g_id, &start, &len, &real);
    ys.assign(len, 0.0f);
    for (uint64_t q = 0; q < real; ++q) {
      uint64_t k = start + q;
      float z = 0.0f;
      for (uint64_t w = 0; w < L->W; ++w)
        z = z + scales[w * L->nc + g_id] * sgn_of_bit(bits + w * words, k);
      z = z / fW;
      uint64_t l = layer_of(layer_off, nl, k);
      float r = rho ? rho[l] : 1.0f;
      ys[q] = (r * e_s[k]) + z;
    }
    ay.assign(real, 0.0f);
    for (uint64_t q = 0; q < real; ++q) ay[q] = std::fabs(ys[q]);
    float sum = orc_cr_sum(ay.data(), real);
    float sscale = real ? sum / (float)real : 0.0f;
    sscales[g_id] = sscale;
    for (uint64_t q = 0; q < len; ++q) {
      uint64_t k = start + q;
      sbits[k >> 5] &= ~(1u << (k & 31));
      if (q < real) {
        bool b = (ys[q] >= 0.0f);
        if (b) sbits[k >> 5] |= (1u << (k & 31));
        e_s[k] = ys[q] - (sscale * (b ? 1.0f : -1.0f));
      } else {
        e_s[k] = 0.0f;
      }
      if (y_out) y_out[k] = ys[q];
    }
  }
}

void orc_server_reduce(const orc_layout* L, const uint64_t* layer_off,
                       uint64_t nl, const float* rho, const uint32_t* bits,
                       const float* scales, float* e_s, uint32_t* sbits,
                       float* sscales, float* y_out) {
  const uint64_t words = L->n_pad / 32 + ((L->n_pad % 32) ? 1 : 0);
  for (uint64_t wd = 0; wd < words; ++wd) sbits[wd] = 0u;
  orc_server_reduce_range(L, layer_off, nl, rho, bits, scales, e_s, sbits, sscales, y_out, 0,
                          L->nc);
}

// Quantisation-error monitor ([TUT] "监控与诊断": watch the norm of the
// quantisation error; [BLOG] §7: check that the error term stays bounded),
// for the 1-bit compressor: per chunk g,
//   out[g] = CR(e[k]^2 over the chunk's real elements)
// the square of the error's 2-norm on that chunk, summed in the fixed order.
// `e` holds true errors e' (worker or server).  Reading: the pages name the
// monitored quantity only as the error's norm; the squared 2-norm per chunk
// is the quantity that adds up over chunks and needs no square root.
void orc_error_norm(const orc_layout* L, const float* e, float* out) {
  std::vector<float> sq;
  for (uint64_t g_id = 0; g_id < L->nc; ++g_id) {
    uint64_t start, len, real;
    chunk_range(L, g_id, &start, &len, &real);
    sq.assign(real, 0.0f);
    for (uint64_t q = 0; q < real; ++q) sq[q] = e[start + q] * e[start + q];
    out[g_id] = orc_cr_sum(sq.data(), real);
  }
}

// Decompression of the server result ([LAMB] ¶2: the global compressed
// momentum is divided by the same fixed coefficient afterwards):
//   out_k = sscale(chunk(k)) * sign(sbit_k) / sigma_l   (sigma = 1 if NULL)
// Padding entries are 0.  With sigma == NULL no division is done.
void orc_decompress(const orc_layout* L, const uint64_t* layer_off,
                    uint64_t nl, const float* sigma, const uint32_t* sbits,
                    const float* sscales, float* out) {
  for (uint64_t g_id = 0; g_id < L->nc; ++g_id) {
    uint64_t start, len, real;
    chunk_range(L, g_id, &start, &len, &real);
    for (uint64_t q = 0; q < len; ++q) {
      uint64_t k = start + q;
      if (q < real) {
        float M = sscales[g_id] * sgn_of_bit(sbits, k);
        if (sigma) M = M / sigma[layer_of(layer_off, nl, k)];
        out[k] = M;
      } else {
        out[k] = 0.0f;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Update with the frozen variance (1-bit Adam)
// ---------------------------------------------------------------------------
// [LAMB] ¶1: after warmup the denominator sqrt(v_{T_w}) is frozen; [BLOG]
// §2.1 gives the Adam step.  No bias correction and no weight decay (the
// pages show none).  m = sscale*sign(sbit), then
//   p = p - lr * (m / (sqrt(v) + eps))
void orc_adam_update(const orc_layout* L, const uint32_t* sbits,
                     const float* sscales, const float* v, float eps, float lr,
                     float* m, float* p) {
  for (uint64_t g_id = 0; g_id < L->nc; ++g_id) {
    uint64_t start, len, real;
    chunk_range(L, g_id, &start, &len, &real);
    for (uint64_t q = 0; q < len; ++q) {
      uint64_t k = start + q;
      if (q >= real) {
        m[k] = 0.0f;
        continue;
      }
      float mk = sscales[g_id] * sgn_of_bit(sbits, k);
      float d = std::sqrt(v[k]);
      d = d + eps;
      float u = mk / d;
      float t = lr * u;
      m[k] = mk;
      p[k] = p[k] - t;
    }
  }
}

// ---------------------------------------------------------------------------
// 1-bit LAMB after warmup
// ---------------------------------------------------------------------------
// Pass A ([LAMB] ¶1 and ¶2), per real element k of layer l:
//   M   = sscale*sign(sbit);  m_t = M / sigma_l
//   g_t = (m_t - b1*m_{t-1}) / (1 - b1)
//   v_t = b2*v_{t-1} + (1 - b2)*g_t^2          (fresh variance)
//   R_l = max(R_l, v_Tw / v_t)                  (infinity norm of the ratio;
//         a NaN ratio (0/0) is skipped, +Inf is kept)
// m and v_t are updated in place; R must hold 0 on entry.
void orc_lamb_pass_a_range(const orc_layout* L, const uint64_t* layer_off,
                           uint64_t nl, const float* sigma, const uint32_t* sbits,
                           const float* sscales, const float* v_frozen, float b1,
                           float b2, float* m, float* v_fresh, float* R, uint64_t g0,
                           uint64_t g1) {
  const float ob1 = 1.0f - b1, ob2 = 1.0f - b2;
  for (uint64_t g_id = g0; g_id < g1 && g_id < L->nc; ++g_id) {
    uint64_t start, len, real;
    chunk_range(L, g_id, &start, &len, &real);
    for (uint64_t q = 0; q < len; ++q) {
      uint64_t k = start + q;
      if (q >= real) {
        m[k] = 0.0f;
        continue;
      }
      uint64_t l = layer_of(layer_off, nl, k);
      float M = sscales[g_id] * sgn_of_bit(sbits, k);
      float mt = M / sigma[l];
      float gt = (mt - (b1 * m[k])) / ob1;
      float vt = (b2 * v_fresh[k]) + (ob2 * (gt * gt));
      m[k] = mt;
      v_fresh[k] = vt;
      float ratio = v_frozen[k] / vt;
      if (!std::isnan(ratio) && ratio > R[l]) R[l] = ratio;
    }
  }
}

void orc_lamb_pass_a(const orc_layout* L, const uint64_t* layer_off,
                     uint64_t nl, const float* sigma, const uint32_t* sbits,
                     const float* sscales, const float* v_frozen, float b1,
                     float b2, float* m, float* v_fresh, float* R) {
  orc_lamb_pass_a_range(L, layer_off, nl, sigma, sbits, sscales, v_frozen, b1, b2, m, v_fresh,
                        R, 0, L->nc);
}

static float fmax_plain(float a, float b) { return a > b ? a : b; }
static float fmin_plain(float a, float b) { return a < b ? a : b; }

// Per-layer ratio and coefficient ([LAMB] ¶1 and ¶3):
//   r_t = clip(clip(R_l, (1-r_thr) r_{t-1}, (1+r_thr) r_{t-1}), r_min, r_max)
//   c_t = clip(c_avg * r_t, c_min, c_max)       (gamma_t in [gamma_min, gamma_max])
//   c_{t-2} <- c_{t-1}; c_{t-1} <- c_t; r_{t-1} <- r_t
// With `frozen` != 0 the ratio is held at 1 and c_t = c_avg ("LAMB + basic
// 1-bit" of ¶1).  c_out receives c_t.
void orc_lamb_ratio(uint64_t nl, const float* R, float r_thr, float r_min,
                    float r_max, float c_min, float c_max, int frozen,
                    const float* c_avg, float* r_prev, float* c_prev,
                    float* c_prev2, float* c_out) {
  for (uint64_t l = 0; l < nl; ++l) {
    float r;
    if (frozen) {
      r = 1.0f;
    } else {
      float lo = (1.0f - r_thr) * r_prev[l];
      float hi = (1.0f + r_thr) * r_prev[l];
      r = fmin_plain(fmax_plain(R[l], lo), hi);
      r = fmin_plain(fmax_plain(r, r_min), r_max);
    }
    float c = c_avg[l] * r;
    c = fmin_plain(fmax_plain(c, c_min), c_max);
    c_prev2[l] = c_prev[l];
    c_prev[l] = c;
    r_prev[l] = r;
    c_out[l] = c;
  }
}

// Step-ratio factor of the error feedback ([LAMB] ¶3: the error carried
// into step t is scaled by c_{t-2}/c_{t-1}); one fp32 division per layer.
void orc_lamb_rho(uint64_t nl, const float* c_prev2, const float* c_prev,
                  float* rho) {
  for (uint64_t l = 0; l < nl; ++l) rho[l] = c_prev2[l] / c_prev[l];
}

// Pass B ([LAMB] ¶1, frozen denominator sqrt(v_Tw)):
//   p = p - (lr*c_l) * (m_t / (sqrt(v_Tw) + eps))
void orc_lamb_pass_b_range(const orc_layout* L, const uint64_t* layer_off,
                           uint64_t nl, const float* c, const float* m,
                           const float* v_frozen, float eps, float lr, float* p,
                           uint64_t g0, uint64_t g1) {
  for (uint64_t g_id = g0; g_id < g1 && g_id < L->nc; ++g_id) {
    uint64_t start, len, real;
    chunk_range(L, g_id, &start, &len, &real);
    for (uint64_t q = 0; q < real; ++q) {
      uint64_t k = start + q;
      uint64_t l = layer_of(layer_off, nl, k);
      float t1 = lr * c[l];
      float d = std::sqrt(v_frozen[k]) + eps;
      float u = m[k] / d;
      p[k] = p[k] - (t1 * u);
    }
  }
}

void orc_lamb_pass_b(const orc_layout* L, const uint64_t* layer_off,
                     uint64_t nl, const float* c, const float* m,
                     const float* v_frozen, float eps, float lr, float* p) {
  orc_lamb_pass_b_range(L, layer_off, nl, c, m, v_frozen, eps, lr, p, 0, L->nc);
}

// ---------------------------------------------------------------------------
// Warmup: uncompressed steps ([BLOG] §6 and [TUT] "预热训练": the first steps
// run at full precision; [LAMB] ¶1: v is frozen at the end of warmup and
// c_avg is the warmup average of LAMB's coefficient)
// ---------------------------------------------------------------------------
// g_bar = (sum over w in order, from 0, of g_w) / W
// m = b1*m + (1-b1)*g_bar;  v = b2*v + (1-b2)*g_bar^2
// Adam (mode 0): p = p - lr*(m/(sqrt(v)+eps))
// LAMB (mode 1): u = m/(sqrt(v)+eps); per layer
//     c = clip(||p_l|| / ||u_l||, c_min, c_max)   (c = 1 if either norm is 0)
//     p = p - (lr*c)*u;  c_sum[l] += c
// Norms are sqrt(CR(x^2)) over the layer, tiles counted from the layer's
// start.  Reading: LAMB's coefficient is the standard trust ratio, clipped;
// the pages name it only as "LAMB's scaling coefficient".
// grads: W pointers, each to n_pad floats.
void orc_warmup_step(const orc_layout* L, const uint64_t* layer_off,
                     uint64_t nl, const float* const* grads, int mode,
                     float b1, float b2, float eps, float lr, float c_min,
                     float c_max, float* m, float* v, float* p, float* c_sum,
                     float* c_out) {
  const float ob1 = 1.0f - b1, ob2 = 1.0f - b2;
  const float fW = (float)L->W;
  std::vector<float> u(L->n, 0.0f);
  for (uint64_t k = 0; k < L->n; ++k) {
    float gb = 0.0f;
    for (uint64_t w = 0; w < L->W; ++w) gb = gb + grads[w][k];
    gb = gb / fW;
    m[k] = (b1 * m[k]) + (ob1 * gb);
    v[k] = (b2 * v[k]) + (ob2 * (gb * gb));
    float d = std::sqrt(v[k]) + eps;
    u[k] = m[k] / d;
    if (mode == 0) p[k] = p[k] - (lr * u[k]);
  }
  for (uint64_t k = L->n; k < L->n_pad; ++k) m[k] = 0.0f;
  if (mode == 0) return;
  uint64_t L_count = nl ? nl : 1;
  std::vector<float> sq;
  for (uint64_t l = 0; l < L_count; ++l) {
    uint64_t a = nl ? layer_off[l] : 0, b = nl ? layer_off[l + 1] : L->n;
    sq.assign(b - a, 0.0f);
    for (uint64_t k = a; k < b; ++k) sq[k - a] = p[k] * p[k];
    float np_ = std::sqrt(orc_cr_sum(sq.data(), b - a));
    for (uint64_t k = a; k < b; ++k) sq[k - a] = u[k] * u[k];
    float nu_ = std::sqrt(orc_cr_sum(sq.data(), b - a));
    float c;
    if (np_ == 0.0f || nu_ == 0.0f) {
      c = 1.0f;
    } else {
      c = np_ / nu_;
      c = fmin_plain(fmax_plain(c, c_min), c_max);
    }
    float t1 = lr * c;
    for (uint64_t k = a; k < b; ++k) p[k] = p[k] - (t1 * u[k]);
    c_sum[l] = c_sum[l] + c;
    if (c_out) c_out[l] = c;
  }
}

// End of warmup for 1-bit LAMB ([LAMB] ¶1, ¶2):
//   rms_l = sqrt(CR(m^2 over layer)) / sqrt(n_l)
//   s_l   = mean_l(rms_l) / rms_l   (s_l = 1 if rms_l == 0); the mean is the
//           in-order sum from 0 divided by the layer count
//   c_avg = c_sum / T_w;  r_prev = 1;  c_prev = c_prev2 = c_avg
// Reading: "a fixed per-layer momentum scale coefficient from the average
// momentum norm" is taken as the factor that brings every layer's momentum
// RMS to the mean RMS over layers; it is not clipped.
void orc_lamb_begin(const orc_layout* L, const uint64_t* layer_off,
                    uint64_t nl, const float* m, const float* c_sum,
                    uint64_t warmup_steps, float* s, float* c_avg,
                    float* r_prev, float* c_prev, float* c_prev2) {
  uint64_t L_count = nl ? nl : 1;
  std::vector<float> rms(L_count, 0.0f), sq;
  for (uint64_t l = 0; l < L_count; ++l) {
    uint64_t a = nl ? layer_off[l] : 0, b = nl ? layer_off[l + 1] : L->n;
    sq.assign(b - a, 0.0f);
    for (uint64_t k = a; k < b; ++k) sq[k - a] = m[k] * m[k];
    float nrm = std::sqrt(orc_cr_sum(sq.data(), b - a));
    rms[l] = nrm / std::sqrt((float)(b - a));
  }
  float mean = 0.0f;
  for (uint64_t l = 0; l < L_count; ++l) mean = mean + rms[l];
  mean = mean / (float)L_count;
  for (uint64_t l = 0; l < L_count; ++l) {
    s[l] = (rms[l] == 0.0f) ? 1.0f : mean / rms[l];
    float ca = c_sum[l] / (float)warmup_steps;
    c_avg[l] = ca;
    r_prev[l] = 1.0f;
    c_prev[l] = ca;
    c_prev2[l] = ca;
  }
}

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
// easy as 1, 2, 3", SC'11): 10 rounds of
//   (c0,c1,c2,c3) -> (hi(M1*c2) ^ c1 ^ k0, lo(M1*c2), hi(M0*c0) ^ c3 ^ k1, lo(M0*c0))
// with M0 = 0xD2511F53, M1 = 0xCD9E8D57, and the key advanced by the Weyl
// constants (0x9E3779B9, 0xBB67AE85) between rounds.
// ---------------------------------------------------------------------------
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2],
                       uint32_t out[4]) {
  uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    uint64_t p0 = (uint64_t)0xD2511F53u * (uint64_t)c0;
    uint64_t p1 = (uint64_t)0xCD9E8D57u * (uint64_t)c2;
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n1 = lo1;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    uint32_t n3 = lo0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

// The uniform used for element k of quantizer call `step`:
// key = (seed low 32, seed high 32),
// counter = (k>>2 low 32, k>>2 high 32, step low 32, step high 32),
// word k & 3 of the output; u = (word >> 8) * 2^-24, an exact float in
// [0, 1).  (The same counter split as a generator started at subsequence
// `step` and offset k.)  Reading: the pages draw "ε ~ U(0,1)" per element
// without naming a generator; Philox is the counter-based generator both
// sides implement.
float orc_uniform(uint64_t seed, uint64_t step, uint64_t k) {
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint64_t grp = k >> 2;
  uint32_t ctr[4] = {(uint32_t)grp, (uint32_t)(grp >> 32), (uint32_t)step,
                     (uint32_t)(step >> 32)};
  uint32_t out[4];
  orc_philox4x32_10(ctr, key, out);
  uint32_t wd = out[k & 3];
  return (float)(wd >> 8) * (1.0f / 16777216.0f);
}

// ---------------------------------------------------------------------------
// Block-wise INT8 stochastic-rounding quantizer ([TUT] "FP32 → INT8 量化"
// and the GradientQuantizeINT8 example)
// ---------------------------------------------------------------------------
// Per block of `block` elements (the last may be short):
//   mx = max |g|  (a NaN never wins the comparison);  scale = mx / 127
//   mx == 0: q = 0 and scale = 0
//   else x = g/scale; f = floor(x); frac = x - f; q = f + (u < frac ? 1 : 0)
//        clamped to [-127, 127]
// deq (optional) = q * scale.  Reading: the example's "floor + Bernoulli"
// form is used (not floor(x + eps)); the two agree in distribution.
// orc_quant_int8_at quantises g[0..n) as the elements k0 .. k0+n-1 of a
// larger tensor (k0 a multiple of `block`): blocks and uniforms are those of
// the whole tensor.  orc_quant_int8 is the whole tensor (k0 = 0).
void orc_quant_int8_at(const float* g, uint64_t n, uint64_t k0, uint64_t block,
                       uint64_t seed, uint64_t step, int8_t* q, float* block_scales,
                       float* deq);

void orc_quant_int8(const float* g, uint64_t n, uint64_t block, uint64_t seed,
                    uint64_t step, int8_t* q, float* block_scales, float* deq) {
  orc_quant_int8_at(g, n, 0, block, seed, step, q, block_scales, deq);
}

void orc_quant_int8_at(const float* g, uint64_t n, uint64_t k0, uint64_t block,
                       uint64_t seed, uint64_t step, int8_t* q, float* block_scales,
                       float* deq) {
  for (uint64_t b0 = 0, bi = 0; b0 < n; b0 += block, ++bi) {
    uint64_t b1 = b0 + block < n ? b0 + block : n;
    float mx = 0.0f;
    for (uint64_t k = b0; k < b1; ++k) {
      float a = std::fabs(g[k]);
      if (a > mx) mx = a;
    }
    if (mx == 0.0f) {
      block_scales[bi] = 0.0f;
      for (uint64_t k = b0; k < b1; ++k) {
        q[k] = 0;
        if (deq) deq[k] = 0.0f;
      }
      continue;
    }
    float scale = mx / 127.0f;
    block_scales[bi] = scale;
    for (uint64_t k = b0; k < b1; ++k) {
      float x = g[k] / scale;
      float f = std::floor(x);
      float frac = x - f;
      float u = orc_uniform(seed, step, k0 + k);
      float qf = f + ((u < frac) ? 1.0f : 0.0f);
      if (qf > 127.0f) qf = 127.0f;
      if (qf < -127.0f) qf = -127.0f;
      if (qf != qf) qf = 0.0f;  // a NaN input codes as 0 (reading)
      q[k] = (int8_t)qf;
      if (deq) deq[k] = qf * scale;
    }
  }
}

// INT8 with error feedback ([TUT] "1-bit 梯度量化" error feedback and
// "精度恢复技巧": keep the residual and add it before the next quantisation;
// applied to the INT8 quantizer of "FP32 → INT8 量化"):
//   x = g + e;  per block of 256: scale = max|x|/127 (0 if max is 0),
//   q = stochastic rounding of x/scale as above;  e' = x - q*scale
// Monitor ([TUT] "监控与诊断": the norm of the quantisation error): err2 (if
// not NULL) receives per block the sum of e'^2 in a fixed order -- lane j
// of 32 adds the squares of elements 4j+c, then 128+4j+c (c = 0..3) from 0,
// then the 32 lane sums meet in a butterfly (v[l] + v[l^o], o = 16..1).
// g, e, q, deq are the elements k0 .. k0+n-1 of a larger tensor (k0 a
// multiple of 256).
void orc_quant_int8_ef_at(const float* g, float* e, uint64_t n, uint64_t k0,
                          uint64_t seed, uint64_t step, int8_t* q, float* block_scales,
                          float* deq, float* err2) {
  const uint64_t block = 256;
  std::vector<float> x(block);
  for (uint64_t b0 = 0, bi = 0; b0 < n; b0 += block, ++bi) {
    uint64_t b1 = b0 + block < n ? b0 + block : n;
    float mx = 0.0f;
    for (uint64_t k = b0; k < b1; ++k) {
      x[k - b0] = g[k] + e[k];
      float a = std::fabs(x[k - b0]);
      if (a > mx) mx = a;
    }
    float scale = mx == 0.0f ? 0.0f : mx / 127.0f;
    block_scales[bi] = scale;
    for (uint64_t k = b0; k < b1; ++k) {
      float qf = 0.0f;
      if (scale != 0.0f) {
        float xs = x[k - b0] / scale;
        float f = std::floor(xs);
        float frac = xs - f;
        float u = orc_uniform(seed, step, k0 + k);
        qf = f + ((u < frac) ? 1.0f : 0.0f);
        if (qf > 127.0f) qf = 127.0f;
        if (qf < -127.0f) qf = -127.0f;
        if (qf != qf) qf = 0.0f;
      }
      q[k] = (int8_t)qf;
      float dq = qf * scale;
      if (deq) deq[k] = dq;
      e[k] = x[k - b0] - dq;
    }
    if (err2) {
      float lane[32];
      for (int j = 0; j < 32; ++j) {
        float acc = 0.0f;
        for (int h = 0; h < 2; ++h)
          for (int c = 0; c < 4; ++c) {
            uint64_t k = b0 + 128 * h + 4 * j + c;
            if (k < b1) acc = acc + (e[k] * e[k]);
          }
        lane[j] = acc;
      }
      for (int o = 16; o >= 1; o >>= 1) {
        float nv[32];
        for (int l = 0; l < 32; ++l) nv[l] = lane[l] + lane[l ^ o];
        for (int l = 0; l < 32; ++l) lane[l] = nv[l];
      }
      err2[bi] = lane[0];
    }
  }
}

// ---------------------------------------------------------------------------
// Layerwise mixed bit widths
// ---------------------------------------------------------------------------
// [BLOG] §3.2 (混合精度训练策略) gives each parameter type its own bit width
// and update period: embeddings and transformer FFN weights 1 bit every
// step, CNN weights 2 bits every step, LayerNorm parameters FP16 every 10
// steps; §6 repeats it as layerwise_bits [1, 2, 1, 16].  [TUT]
// "更激进的组合策略" (分层混合精度) names the same idea.  Neither page
// defines the 2-bit code or what happens between two FP16 updates.
// Readings:
//   - the layers of one width form a fused buffer of their own, with the
//     layout above (n = that group's elements), compressed by one codec;
//     width 1 is the scaled sign above;
//   - width b in {2, 4, 8} is the b-bit form of [TUT]'s quantizer, whose
//     GradientQuantizeINT8 example takes the width as an argument: per block
//     of 256 elements scale = max|x| / (2^(b-1) - 1) (0 if the max is 0),
//     stochastic rounding as in the INT8 quantizer, clamp to
//     [-(2^(b-1) - 1), 2^(b-1) - 1], a NaN codes as 0, and error feedback
//     e' = x - q*scale.  b = 2 gives the codes -1, 0, 1.  Blocks are counted
//     over each worker's whole buffer (block k/256); the alignment A is a
//     multiple of 256, so no block straddles two partitions and the server's
//     blocks are the workers' blocks;
//   - the uniform of worker w's element k is orc_uniform(seed, step,
//     w*n_pad + k), that of the server's element k orc_uniform(seed, step,
//     W*n_pad + k): the element's index in the W+1 messages laid end to end;
//   - width 16 sends x as IEEE binary16 (round to nearest, ties to even)
//     with error feedback e' = x - f32(h), on the steps where `send` is set
//     (every 10th).  On the other steps nothing is exchanged: each worker
//     keeps x whole as its error, the server keeps its error, the momentum
//     is 0 and the parameters are left as they are;
//   - 1-bit Adam only (the table sits in the 1bit Adam write-up); no sigma,
//     no rho.
// Codes: the field q mod 2^b of element k sits at bit (k*b) % 32 of word
// (k*b)/32 (LSB first, two's complement); a row holds n_pad*b/32 words.
// The *_at functions take the elements [k0, k0+len) of the buffer (k0 and
// len multiples of 256): the arrays passed hold just that range (codes from
// word k0*b/32, scales from block k0/256), so that a sample of blocks can be
// checked on its own.  Elements k >= n are padding: code 0, error 0, m 0.

static void qb_put(uint32_t* words, uint64_t k, int bits, int q) {
  const uint64_t bit = k * (uint64_t)bits;
  const uint32_t field = (uint32_t)q & ((1u << bits) - 1u);
  words[bit / 32] |= field << (bit % 32);
}

static int qb_get(const uint32_t* words, uint64_t k, int bits) {
  const uint64_t bit = k * (uint64_t)bits;
  const int field = (int)((words[bit / 32] >> (bit % 32)) & ((1u << bits) - 1u));
  return field >= (1 << (bits - 1)) ? field - (1 << bits) : field;
}

// Quantises the block of 256 values x[0..256) that are the elements
// kb .. kb+255 of a buffer of n real elements; `u_base` + k is the uniform's
// element index; codes are relative to the block's own first element (the
// caller passes the row's words from that block on).
static void qb_block(int bits, uint64_t n, uint64_t kb, const float* x, uint64_t seed,
                     uint64_t step, uint64_t u_base, uint32_t* codes, float* scale_out,
                     float* e) {
  const float qmax = (float)((1 << (bits - 1)) - 1);
  float mx = 0.0f;
  for (uint64_t i = 0; i < 256; ++i) {
    if (kb + i >= n) break;
    float a = std::fabs(x[i]);
    if (a > mx) mx = a;  // a NaN never wins
  }
  const float scale = mx == 0.0f ? 0.0f : mx / qmax;
  *scale_out = scale;
  for (uint64_t i = 0; i < 256; ++i) {
    const uint64_t k = kb + i;
    if (k >= n) {
      e[i] = 0.0f;
      continue;
    }
    float qf = 0.0f;
    if (scale != 0.0f) {
      float xs = x[i] / scale;
      float f = std::floor(xs);
      float frac = xs - f;
      float u = orc_uniform(seed, step, u_base + k);
      qf = f + ((u < frac) ? 1.0f : 0.0f);
      if (qf > qmax) qf = qmax;
      if (qf < -qmax) qf = -qmax;
      if (qf != qf) qf = 0.0f;
    }
    qb_put(codes, i, bits, (int)qf);
    e[i] = x[i] - (qf * scale);
  }
}

// Worker w, b-bit codec:
//   m_w = b1*m + (1-b1)*g;  x = m_w + e  (clamped to [-clip, clip] if clip > 0)
//   per block: the quantizer above;  e := x - q*scale (plain, not deferred)
// codes: the worker's row from word k0*b/32; bscales from block k0/256.
void orc_qb_compress_worker_at(const orc_layout* L, int bits, float b1, float clip,
                               uint64_t w, uint64_t seed, uint64_t step, uint64_t k0,
                               uint64_t len, const float* g, const float* m, float* e,
                               uint32_t* codes, float* bscales) {
  const float ob1 = 1.0f - b1;
  const uint64_t words = len * (uint64_t)bits / 32;
  for (uint64_t i = 0; i < words; ++i) codes[i] = 0u;
  std::vector<float> x(256);
  for (uint64_t b0 = 0; b0 < len; b0 += 256) {
    for (uint64_t i = 0; i < 256; ++i) {
      const uint64_t k = k0 + b0 + i;
      if (k >= L->n) {
        x[i] = 0.0f;
        continue;
      }
      float mw = (b1 * m[b0 + i]) + (ob1 * g[b0 + i]);
      float xv = mw + e[b0 + i];
      if (clip > 0.0f) {
        if (xv > clip) xv = clip;
        if (xv < -clip) xv = -clip;
      }
      x[i] = xv;
    }
    qb_block(bits, L->n, k0 + b0, x.data(), seed, step, w * L->n_pad,
             codes + b0 * (uint64_t)bits / 32, &bscales[b0 / 256], e + b0);
  }
}

void orc_qb_compress_worker(const orc_layout* L, int bits, float b1, float clip, uint64_t w,
                            uint64_t seed, uint64_t step, const float* g, const float* m,
                            float* e, uint32_t* codes, float* bscales) {
  orc_qb_compress_worker_at(L, bits, b1, clip, w, seed, step, 0, L->n_pad, g, m, e, codes,
                            bscales);
}

// Server, b-bit codec, elements [k0, k0+len) of every partition it covers:
//   z = (sum over w = 0..W-1, in order, from 0, of q_w*scale_w) / W
//   y = e_s + z;  per block the quantizer above;  e_s := y - q_s*sscale
// codes: W rows of `row_words` words, each from word k0*b/32 of its row;
// bscales: W rows of `row_blocks` scales, each from block k0/256.
void orc_qb_server_at(const orc_layout* L, int bits, uint64_t seed, uint64_t step,
                      uint64_t k0, uint64_t len, const uint32_t* codes, uint64_t row_words,
                      const float* bscales, uint64_t row_blocks, float* e_s,
                      uint32_t* scodes, float* sbscales) {
  const float fW = (float)L->W;
  const uint64_t words = len * (uint64_t)bits / 32;
  for (uint64_t i = 0; i < words; ++i) scodes[i] = 0u;
  std::vector<float> y(256);
  for (uint64_t b0 = 0; b0 < len; b0 += 256) {
    for (uint64_t i = 0; i < 256; ++i) {
      const uint64_t k = k0 + b0 + i;
      if (k >= L->n) {
        y[i] = 0.0f;
        continue;
      }
      float z = 0.0f;
      for (uint64_t w = 0; w < L->W; ++w) {
        const float q = (float)qb_get(codes + w * row_words, b0 + i, bits);
        z = z + (q * bscales[w * row_blocks + b0 / 256]);
      }
      z = z / fW;
      y[i] = e_s[b0 + i] + z;
    }
    qb_block(bits, L->n, k0 + b0, y.data(), seed, step, L->W * L->n_pad,
             scodes + b0 * (uint64_t)bits / 32, &sbscales[b0 / 256], e_s + b0);
  }
}

void orc_qb_server(const orc_layout* L, int bits, uint64_t seed, uint64_t step,
                   const uint32_t* codes, const float* bscales, float* e_s, uint32_t* scodes,
                   float* sbscales) {
  orc_qb_server_at(L, bits, seed, step, 0, L->n_pad, codes, L->n_pad * (uint64_t)bits / 32,
                   bscales, L->n_pad / 256, e_s, scodes, sbscales);
}

// out = q*scale (padding 0), elements [k0, k0+len).
void orc_qb_decode_at(const orc_layout* L, int bits, uint64_t k0, uint64_t len,
                      const uint32_t* codes, const float* bscales, float* out) {
  for (uint64_t i = 0; i < len; ++i) {
    if (k0 + i >= L->n) {
      out[i] = 0.0f;
      continue;
    }
    out[i] = (float)qb_get(codes, i, bits) * bscales[i / 256];
  }
}

// 1-bit Adam update fed by the b-bit server message (frozen variance, as
// orc_adam_update): m = q*sscale;  p = p - lr*(m/(sqrt(v) + eps)).
void orc_qb_adam_at(const orc_layout* L, int bits, float eps, float lr, uint64_t k0,
                    uint64_t len, const uint32_t* scodes, const float* sbscales,
                    const float* v, float* m, float* p) {
  for (uint64_t i = 0; i < len; ++i) {
    if (k0 + i >= L->n) {
      m[i] = 0.0f;
      continue;
    }
    float mk = (float)qb_get(scodes, i, bits) * sbscales[i / 256];
    float d = std::sqrt(v[i]);
    d = d + eps;
    float u = mk / d;
    float t = lr * u;
    m[i] = mk;
    p[i] = p[i] - t;
  }
}

// IEEE 754 binary16 from binary32, round to nearest, ties to even, written
// from the format's definition: 1 sign bit, 5 exponent bits (bias 15), 10
// fraction bits; normal values 2^-14 .. 65504, subnormal steps of 2^-24.
// A value is rounded to a multiple of its binade's step (2^(e-10) for
// 2^e <= |x| < 2^(e+1), 2^-24 below 2^-14); |x| >= 65520 (65504 plus half a
// step, which rounds up to 2^16) becomes infinity.  A NaN becomes the quiet
// NaN 0x7e00 with the input's sign.
uint16_t orc_f32_to_f16(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  const uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
  const double a = std::fabs((double)f);
  if (f != f) return (uint16_t)(sign | 0x7e00u);
  if (a >= 65520.0) return (uint16_t)(sign | 0x7c00u);
  int e2;
  std::frexp(a, &e2);  // a = mant * 2^e2, mant in [0.5, 1): 2^(e2-1) <= a < 2^e2
  const int e = e2 - 1;
  const bool sub = (a < std::ldexp(1.0, -14));
  const double step = sub ? std::ldexp(1.0, -24) : std::ldexp(1.0, e - 10);
  const double r = std::nearbyint(a / step);  // exact quotient; ties to even
  if (sub) return (uint16_t)(sign | (uint16_t)r);  // r = 1024 is 2^-14, normal
  // r in [1024, 2048]; r = 2048 carries into the next binade by itself
  return (uint16_t)(sign | (uint16_t)(((e + 15) << 10) + ((int)r - 1024)));
}

float orc_f16_to_f32(uint16_t h) {
  const int s = (h >> 15) & 1, ex = (h >> 10) & 31, fr = h & 1023;
  double v;
  if (ex == 0) v = std::ldexp((double)fr, -24);
  else if (ex == 31) v = fr ? NAN : INFINITY;
  else v = std::ldexp((double)(1024 + fr), ex - 25);
  return (float)(s ? -v : v);
}

// Worker, FP16 codec (elements [0, n_pad)):
//   x = m_w + e (clamped if clip > 0);
//   send:  h = f16(x), e := x - f32(h);   otherwise: e := x, h untouched.
void orc_f16_compress_worker(const orc_layout* L, float b1, float clip, int send,
                             const float* g, const float* m, float* e, uint16_t* h) {
  const float ob1 = 1.0f - b1;
  for (uint64_t k = 0; k < L->n_pad; ++k) {
    if (k >= L->n) {
      e[k] = 0.0f;
      if (send) h[k] = 0;
      continue;
    }
    float mw = (b1 * m[k]) + (ob1 * g[k]);
    float x = mw + e[k];
    if (clip > 0.0f) {
      if (x > clip) x = clip;
      if (x < -clip) x = -clip;
    }
    if (send) {
      const uint16_t hk = orc_f32_to_f16(x);
      h[k] = hk;
      e[k] = x - orc_f16_to_f32(hk);
    } else {
      e[k] = x;
    }
  }
}

// Server, FP16 codec, on a sending step: h is [W][n_pad];
//   z = (sum over w, in order, from 0, of f32(h_w)) / W;  y = e_s + z
//   hs = f16(y);  e_s := y - f32(hs)
void orc_f16_server(const orc_layout* L, const uint16_t* h, float* e_s, uint16_t* hs) {
  const float fW = (float)L->W;
  for (uint64_t k = 0; k < L->n_pad; ++k) {
    if (k >= L->n) {
      e_s[k] = 0.0f;
      hs[k] = 0;
      continue;
    }
    float z = 0.0f;
    for (uint64_t w = 0; w < L->W; ++w) z = z + orc_f16_to_f32(h[w * L->n_pad + k]);
    z = z / fW;
    const float y = e_s[k] + z;
    const uint16_t hk = orc_f32_to_f16(y);
    hs[k] = hk;
    e_s[k] = y - orc_f16_to_f32(hk);
  }
}

// Update, FP16 codec: sending step m = f32(hs), p = p - lr*(m/(sqrt(v)+eps));
// other steps m = 0 and p is left as it is.  Padding: m = 0.
void orc_f16_adam(const orc_layout* L, int send, float eps, float lr, const uint16_t* hs,
                  const float* v, float* m, float* p) {
  for (uint64_t k = 0; k < L->n_pad; ++k) {
    if (k >= L->n || !send) {
      m[k] = 0.0f;
      continue;
    }
    float mk = orc_f16_to_f32(hs[k]);
    float d = std::sqrt(v[k]);
    d = d + eps;
    float u = mk / d;
    float t = lr * u;
    m[k] = mk;
    p[k] = p[k] - t;
  }
}

}  // extern "C"
