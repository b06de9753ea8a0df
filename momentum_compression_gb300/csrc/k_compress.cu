// Worker compression of the 1-bit compressed optimizer step, all W workers
// in one pass over the fused buffer.
//
// Per element k of worker w ("1bit Adam" write-up, 2.1; gradient
// quantization tutorial, "1-bit 梯度量化"; 1-bit LAMB summary, paragraphs
// 2-3):
//   e_w   = x_prev - scale_prev*sign(x_prev)   (the deferred error of the
//           previous step, rebuilt from the stored x, bits and scale)
//   m_w   = b1*m + (1-b1)*g_w
//   x     = sigma_l*m_w + rho_l*e_w            (1-bit Adam: m_w + e_w),
//           limited to [-clip, clip] when clip > 0 ("1bit Adam" write-up 4.1)
//   bit   = x >= 0; x is stored in place of e_w
//   scale(chunk) = mean |x| over the chunk: this kernel writes one total
//   per (worker, tile); k_finalize_scales adds them in tile order
//
// Work decomposition: a CTA owns a sequence of 4096-element tiles and, for
// each, all W workers, so the momentum m is read once per element.  The
// CTA is warp-specialised: one producer thread streams, for every
// (tile, worker) item, the gradient and error tiles into a ring of
// shared-memory stages with cp.async.bulk (completion counted in bytes on
// an mbarrier), and the m tile into its own buffer; eight consumer warps
// take the items in order.  Consumer lane p handles elements
// 1024*i + 4*p + c (i, c = 0..3) -- 128-bit shared-memory reads, and the
// fixed summation order of the tile total.  Signs are packed with three
// xor-shuffles per 32-bit word; the new x goes back to global memory with
// plain 128-bit stores.  No wait is unbounded (ptx.cuh), and no CTA
// ever waits for another.  The copies carry no L2 eviction hint: with an
// evict-first policy on them the kernel measured 1-4% slower.
#include <type_traits>

#include "ob_internal.cuh"
#include "ptx.cuh"

namespace ob {
namespace {

constexpr int kConsumers = kThreads;            // 8 warps
constexpr int kCompressThreads = kThreads + 32;  // + 1 producer warp

// With the momentum in sign form (re-reading it costs 1/8 byte per element)
// a tile's workers are taken in groups of at most kGroup, group-major over
// the buffer: fewer workers' arrays are streamed at once, which measured
// faster (fp32 gradients: compress at W = 3-4 ran at ~98% of the copy peak,
// at W = 8 ~90%; in groups of 4, W = 8 and 16 run at ~97%; groups of 2
// were 14% slower there).  With bf16 gradients groups of 2 measured best
// (GPT-1.3B, W = 4: 3.3% faster than one group of 4, W = 8: 4.5%; groups of
// 1 slower).  With a dense m the groups measured slower (m is re-read per
// group and its single buffer serialises them).
constexpr uint32_t kGroupF32 = 4, kGroupBF16 = 2;

// A stage holds one (tile, worker) item: the gradient tile, the error tile
// and the worker's previous sign words of the tile (a 16-byte aligned run),
// 32.5 KB with fp32 gradients, 24.5 KB with bf16.  Two CTAs per SM, each
// with 2 (fp32) or 3 (bf16) stages plus the m tile, so that 4-6 items are
// in flight per SM; with the momentum in sign form the m tile's room holds
// one more stage.
constexpr uint32_t kRunWords = kTile / 32 + 8;  // one tile's words + rounding slack

template <bool BF16, bool MSIGN>
struct CompressSmem {
  static constexpr int kStages = (BF16 ? 3 : 2) + (MSIGN ? 1 : 0);
  static constexpr uint32_t kG = BF16 ? 2u : 4u;
  static constexpr size_t kStageG = kTile * kG;
  static constexpr size_t kStageE = kTile * 4;
  static constexpr size_t kStageB = kRunWords * 4;
  static constexpr size_t kStage = kStageG + kStageE + kStageB;
  static constexpr size_t kM = MSIGN ? 0 : kTile * 4;
  static constexpr size_t kBars = (2 * kStages + 2) * 8;
  static constexpr size_t kWs = 2 * OB_MAX_WORKERS * 8 * 4;  // warp totals, by tile parity
  static constexpr size_t kSc = 2 * OB_MAX_WORKERS * 4;
  static constexpr size_t kBytes = kM + kStages * kStage + kBars + kWs + kSc;
};

// MSIGN: the momentum is read in its sign form (msscale*sign(msbit), what
// the previous server step produced) instead of as a dense fp32 tile.
template <bool BF16, bool LAMB, bool MSIGN>
__global__ void __launch_bounds__(kCompressThreads, 2) k_compress(const CompressArgs A) {
  using S = CompressSmem<BF16, MSIGN>;
  constexpr int kStages = S::kStages;
  extern __shared__ __align__(128) unsigned char smem[];
  float* mbuf = reinterpret_cast<float*>(smem);  // [4096]
  unsigned char* stage0 = smem + S::kM;
  uint64_t* bars = reinterpret_cast<uint64_t*>(stage0 + kStages * S::kStage);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* mfull = bars + 2 * kStages;
  uint64_t* mempty = bars + 2 * kStages + 1;
  // warp totals [2][OB_MAX_WORKERS][8], double-buffered by tile parity so
  // that one barrier per tile suffices
  float(*ws2)[8] = reinterpret_cast<float(*)[8]>(bars + 2 * kStages + 2);
  // the workers' chunk scales of the current and the next tile
  float(*s_sc)[OB_MAX_WORKERS] =
      reinterpret_cast<float(*)[OB_MAX_WORKERS]>(ws2 + 2 * OB_MAX_WORKERS);
  __shared__ volatile int s_abort;
  // 1-bit LAMB per-tile scalars (first layer, its end, sigma, rho) of the
  // current and the next work item, made by thread 0 an item ahead: the
  // layer of the item after next and the loads that depend on the next
  // item's layer go out by cp.async, so no register and no consumer waits
  // on them (the chain tile -> layer -> sigma, rho used to stall every
  // consumer at each item start).
  struct LMeta {
    uint64_t lend;
    uint32_t l;
    float s, r;
  };
  struct LRaw {
    uint64_t lend;
    uint32_t l, l_next;
    float s, c2, c1;
  };
  __shared__ LMeta s_lm[2];
  __shared__ LRaw s_lr;

  const Geo& G = A.geo;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  unsigned* err = A.ws.err;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumers / 32);
    }
    mbar_init(mfull, 1);
    mbar_init(mempty, kConsumers / 32);
    s_abort = 0;
    fence_barrier_init();
  }
  __syncthreads();

  // work items: (worker group, tile), group-major.  Only 1-bit Adam with
  // the sign-form m takes the workers in groups (fewer worker streams at
  // once measured faster there); a dense m would be re-read per group, and
  // 1-bit LAMB's per-tile layer setup measured slower repeated per group
  constexpr bool kGrouped = MSIGN && !LAMB;
  constexpr uint32_t kGroup = BF16 ? kGroupBF16 : kGroupF32;
  // NW workers are compressed: all W of the layout, or one (a rank's own)
  const uint32_t NW = A.nw;
  const uint32_t gsz = kGrouped ? kGroup : NW;
  const uint32_t n_groups = kGrouped ? (NW + kGroup - 1) / kGroup : 1u;
  const uint32_t n_vt = G.n_tiles * n_groups;

  // ------------------------------------------------------------ producer
  if (warp == kConsumers / 32) {
    if (lane != 0) return;
    uint32_t item = 0, ti = 0;
    bool ok = true;
    for (uint32_t VT = blockIdx.x; ok && VT < n_vt; VT += gridDim.x, ++ti) {
      const uint32_t gi = kGrouped ? VT / G.n_tiles : 0u, T = VT - gi * G.n_tiles;
      const uint32_t wbeg = gi * gsz, wend = wbeg + gsz < NW ? wbeg + gsz : NW;
      const Tile tl = decode_tile(G, T);
      if constexpr (!MSIGN) {
        if (ti >= 1) ok = mbar_wait(mempty, (ti - 1) & 1, err, kErrWaitEmpty);
        if (!ok || s_abort) break;
        mbar_arrive_expect_tx(mfull, tl.len * 4);
        bulk_g2s(mbuf, A.m + tl.start, tl.len * 4, mfull);
      }
      for (uint32_t w = wbeg; w < wend; ++w, ++item) {
        const uint32_t s = item % kStages, r = item / kStages;
        if (r >= 1) ok = mbar_wait(&empty[s], (r - 1) & 1, err, kErrWaitEmpty);
        if (!ok || s_abort) {
          ok = false;
          break;
        }
        unsigned char* st = stage0 + s * S::kStage;
        // the previous words of (tile, worker): only this CTA rewrites them,
        // after this copy has landed; the rounding words are not used
        const uint64_t w0 = (tl.start >> 5) & ~uint64_t(3);
        const uint32_t run = (uint32_t)((((tl.start + tl.len) / 32 + 3) & ~uint64_t(3)) - w0) * 4;
        mbar_arrive_expect_tx(&full[s], tl.len * (S::kG + 4) + run);
        bulk_g2s(st, static_cast<const unsigned char*>(A.g[w]) + tl.start * S::kG,
                        tl.len * S::kG, &full[s]);
        bulk_g2s(st + S::kStageG, A.e[w] + tl.start, tl.len * 4, &full[s]);
        bulk_g2s(st + S::kStageG + S::kStageE, A.bits + (uint64_t)w * G.words + w0, run,
                 &full[s]);
      }
    }
    if (!ok) s_abort = 1;
    // Drain: every copy this thread issued must have landed before exit.
    for (uint32_t k = 0; k < kStages && k < item; ++k) {
      const uint32_t it = item - 1 - k;
      if (!mbar_wait(&full[it % kStages], (it / kStages) & 1, err, kErrDrain)) break;
    }
    if (!MSIGN && ti >= 1) mbar_wait(mfull, (ti - 1) & 1, err, kErrDrain);
    return;
  }

  // ------------------------------------------------------------ consumers
  const float b1 = A.b1, ob1 = A.ob1, clip = A.clip;
  const int p = tid;
  // MSIGN: the momentum's sign words and chunk scale of the next tile are
  // loaded one tile ahead, so their latency hides behind the current tile
  uint32_t mw_next[4] = {0u, 0u, 0u, 0u};
  float mss_next = 0.0f;
  auto load_msign = [&](const Tile& tn) {
    mss_next = __ldcg(A.msscales + tn.g);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t off = 1024u * i + 4u * p;
      mw_next[i] = off < tn.len ? __ldg(A.msbits + ((tn.start + off) >> 5)) : 0u;
    }
  };
  // tile of work item V
  auto tile_of = [&](uint32_t V) { return kGrouped ? V % G.n_tiles : V; };
  if constexpr (LAMB) {
    if (p == 0 && blockIdx.x < n_vt) {
      const uint32_t T0 = tile_of(blockIdx.x);
      const uint32_t l = __ldg(A.ws.tile_layer + T0);
      s_lm[0].l = l;
      s_lm[0].lend = __ldg(A.ws.layer_off + l + 1);
      s_lm[0].s = __ldg(A.s + l);
      s_lm[0].r = A.ratio_ef ? __fdiv_rn(__ldg(A.c_prev2 + l), __ldg(A.c_prev + l)) : 1.0f;
      if (blockIdx.x + gridDim.x < n_vt) {
        cp_async_4(&s_lr.l_next, A.ws.tile_layer + tile_of(blockIdx.x + gridDim.x));
        cp_async_commit();
        cp_async_wait_all();
      }
    }
  }
  if (blockIdx.x < n_vt) {
    const uint32_t gi = kGrouped ? blockIdx.x / G.n_tiles : 0u, T0 = blockIdx.x - gi * G.n_tiles;
    const Tile t0 = decode_tile(G, T0);
    if constexpr (MSIGN) load_msign(t0);
    const uint32_t wb = gi * gsz, nw = (wb + gsz < NW ? wb + gsz : NW) - wb;
    if ((uint32_t)p < nw) s_sc[0][p] = __ldcg(A.scales + (uint64_t)(wb + p) * G.nc + t0.g);
  }
  named_sync(1, kConsumers);
  uint32_t item = 0, ti = 0;
  for (uint32_t VT = blockIdx.x; VT < n_vt; VT += gridDim.x, ++ti) {
    const uint32_t gi = kGrouped ? VT / G.n_tiles : 0u, T = VT - gi * G.n_tiles;
    const uint32_t wbeg = gi * gsz, wend = wbeg + gsz < NW ? wbeg + gsz : NW;
    const Tile tl = decode_tile(G, T);
    float(*ws)[8] = ws2 + (ti & 1) * OB_MAX_WORKERS;
    bool ok = true;
    // MSIGN: this tile's momentum words and scale, taken before the next
    // tile's are loaded over them
    [[maybe_unused]] uint32_t mnib[4];
    [[maybe_unused]] float mss = 0.0f;
    if constexpr (MSIGN) {
      mss = mss_next;
#pragma unroll
      for (int i = 0; i < 4; ++i) mnib[i] = mw_next[i] >> (4 * (p & 7));
    }
    // the next item group: its tile, decoded once, for its worker scales
    // (stored before this group's barrier) and its momentum words
    float sc_next = 0.0f;
    const uint32_t VTn = VT + gridDim.x;
    uint32_t nwn = 0;
    if (VTn < n_vt) {
      const uint32_t gin = kGrouped ? VTn / G.n_tiles : 0u;
      const Tile tn = decode_tile(G, VTn - gin * G.n_tiles);
      const uint32_t wbn = gin * gsz;
      nwn = (wbn + gsz < NW ? wbn + gsz : NW) - wbn;
      if ((uint32_t)p < nwn) sc_next = __ldcg(A.scales + (uint64_t)(wbn + p) * G.nc + tn.g);
      if constexpr (MSIGN) load_msign(tn);
    }
    // 1-bit LAMB: the layer of the tile's first element; every worker pass
    // walks the layers forward from it (layers change rarely inside a tile)
    uint32_t l_t = 0;
    uint64_t lend_t = 0;
    float s_t = 1.0f, r_t = 1.0f;
    if constexpr (LAMB) {
      const LMeta& lm = s_lm[ti & 1];
      l_t = lm.l;
      lend_t = lm.lend;
      s_t = lm.s;
      r_t = lm.r;
      if (p == 0 && VTn < n_vt) {
        // the next item's scalars, from its layer loaded an item ago; then
        // the layer of the item after it
        const uint32_t ln = s_lr.l_next;
        s_lr.l = ln;
        cp_async_8(&s_lr.lend, A.ws.layer_off + ln + 1);
        cp_async_4(&s_lr.s, A.s + ln);
        if (A.ratio_ef) {
          cp_async_4(&s_lr.c2, A.c_prev2 + ln);
          cp_async_4(&s_lr.c1, A.c_prev + ln);
        }
        if (VTn + gridDim.x < n_vt)
          cp_async_4(&s_lr.l_next, A.ws.tile_layer + tile_of(VTn + gridDim.x));
        cp_async_commit();
      }
    }
    const bool uni = !LAMB || tl.start + tl.len <= lend_t || G.n <= lend_t;
    // a separate full-tile body only where it fits the registers (bf16
    // gradients with 1-bit Adam: the fp32 and LAMB variants spill with it)
    constexpr bool kFullPath = BF16 && !LAMB;
    const bool full_tile = kFullPath && tl.len == kTile && tl.start + kTile <= G.n;
    // the tile's m in registers, shared by its workers
    float4 mv[4];
    // row i (elements tl.start + 1024i + 4p + c) lies in the tile: padding
    // rows inside the tile are still stored (as 0); an element is a real
    // one if its row is valid and its index is below n.  1-bit LAMB tests
    // the tile offset against a 32-bit limit instead (fewer registers
    // there; for 1-bit Adam the 64-bit index test measured faster).
    bool valid[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) valid[i] = 1024u * i + 4u * p < tl.len;
    [[maybe_unused]] const uint32_t lim =
        !LAMB || G.n <= tl.start ? 0u
                                 : (G.n - tl.start < tl.len ? (uint32_t)(G.n - tl.start) : tl.len);
    auto real = [&](int i, int c, uint64_t k) {
      if constexpr (LAMB) return 1024u * i + 4u * p + c < lim;
      else return valid[i] && k < G.n;
    };
    if constexpr (MSIGN) {
      // m = sscale*sign (1-bit Adam) or sscale*sign/sigma_l (1-bit LAMB);
      // +-sscale/sigma = (+-sscale)/sigma exactly (IEEE division is
      // symmetric in sign): one division per layer
      [[maybe_unused]] uint32_t lq = l_t;
      [[maybe_unused]] uint64_t lqend = lend_t;
      float q = LAMB ? __fdiv_rn(mss, s_t) : mss;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if constexpr (LAMB) {
            const uint64_t k = tl.start + 1024u * i + 4u * p + c;
            if (!uni && real(i, c, k) && advance_layer(A.ws.layer_off, G.L, k, lq, lqend))
              q = __fdiv_rn(mss, __ldg(A.s + lq));
          }
          f4at(mv[i], c) = ((mnib[i] >> c) & 1u) ? q : -q;
        }
      }
    } else {
      ok = s_abort == 0 && mbar_wait(mfull, ti & 1, err, kErrWaitFull);
      if (!ok) s_abort = 1;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t off = 1024u * i + 4u * p;
        mv[i] = valid[i] ? *reinterpret_cast<const float4*>(mbuf + off)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(mempty);
    }


    const uint32_t wshift = (uint32_t)((tl.start >> 5) & 3);  // rounding of the word runs
    for (uint32_t w = wbeg; w < wend; ++w, ++item) {
      const uint32_t s = item % kStages;
      const float osc = s_sc[ti & 1][w - wbeg];
      uint32_t* __restrict__ bw = A.bits + (uint64_t)w * G.words;
      float* __restrict__ e = A.e[w];
      ok = s_abort == 0 && mbar_wait(&full[s], (item / kStages) & 1, err, kErrWaitFull);
      if (!ok) s_abort = 1;
      const unsigned char* st = stage0 + s * S::kStage;
      const uint32_t* sow = reinterpret_cast<const uint32_t*>(st + S::kStageG + S::kStageE);
      // g and e of row i from the stage
      auto fetch = [&](int i, float4& g4, float4& e4) {
        const uint32_t off = 1024u * i + 4u * p;
        if (valid[i]) {
          if constexpr (BF16) {
            const uint2 u = *reinterpret_cast<const uint2*>(st + off * 2);
            g4 = make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                             __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
          } else {
            g4 = *reinterpret_cast<const float4*>(st + off * 4);
          }
          e4 = *reinterpret_cast<const float4*>(st + S::kStageG + off * 4);
        } else {
          g4 = e4 = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      };
      // Early: the whole stage into registers and released at once (fp32
      // gradients, 1-bit Adam, sign-form m).  Late: row by row inside the
      // body and released after it -- the stages still in flight cover the
      // memory latency.  1-bit LAMB needs late release to stay below the
      // spill point; for the dense m and bf16 gradients it measured faster
      // (BERT-base dense 1.80 -> 1.73 ms, GPT-1.3B 9.13 -> 9.01 ms), for
      // the fp32 sign-form path slightly slower (1.646 -> 1.665 ms).
      constexpr bool kLate = LAMB || !MSIGN || BF16;
      [[maybe_unused]] float4 gv[4], ev[4];
      uint32_t owd[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t off = 1024u * i + 4u * p;
        owd[i] = valid[i] ? sow[(off >> 5) + wshift] : 0u;
        if constexpr (!kLate) fetch(i, gv[i], ev[i]);
      }
      if constexpr (!kLate) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);  // the stage is in registers now
      }

      // UNI: the whole tile lies in one layer (sigma, rho scalar); else the
      // layers are walked element by element
      // FULL: all 4096 elements of the tile are real (no per-element checks)
      auto body = [&](auto uni_tag, auto full_tag) -> float {
        [[maybe_unused]] constexpr bool UNI = decltype(uni_tag)::value;
        constexpr bool FULL = decltype(full_tag)::value;
        float acc = 0.0f;
        [[maybe_unused]] uint32_t l = l_t;
        [[maybe_unused]] uint64_t lend = lend_t;
        [[maybe_unused]] float s_l = s_t, r_l = r_t;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint64_t k0 = tl.start + 1024u * i + 4u * p;
          float4 xv, g4, e4;
          if constexpr (kLate) fetch(i, g4, e4);
          else g4 = gv[i], e4 = ev[i];
          uint32_t nib = 0;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            float x = 0.0f;
            if (FULL || real(i, c, k0 + c)) {
              // scale*sign (a test and select: fewer instructions here than
              // flipping the sign bit)
              const float so = ((owd[i] >> (4 * (p & 7) + c)) & 1u) ? osc : -osc;
              const float et = __fsub_rn(f4get(e4, c), so);
              if constexpr (LAMB && !UNI) {
                if (advance_layer(A.ws.layer_off, G.L, k0 + c, l, lend)) {
                  s_l = __ldg(A.s + l);
                  r_l = A.ratio_ef ? __fdiv_rn(__ldg(A.c_prev2 + l), __ldg(A.c_prev + l))
                                   : 1.0f;
                }
              }
              const float mw =
                  __fadd_rn(__fmul_rn(b1, f4get(mv[i], c)), __fmul_rn(ob1, f4get(g4, c)));
              if constexpr (LAMB) {
                x = __fadd_rn(__fmul_rn(s_l, mw), __fmul_rn(r_l, et));
              } else {
                x = __fadd_rn(mw, et);
              }
              if (clip > 0.0f) {  // a NaN stays NaN
                x = x > clip ? clip : x;
                x = x < -clip ? -clip : x;
              }
              acc = __fadd_rn(acc, fabsf(x));
              if (x >= 0.0f) nib |= 1u << c;
            }
            f4at(xv, c) = x;
          }
          const uint32_t word = pack_word(nib, lane);
          if (FULL || valid[i]) {
            *reinterpret_cast<float4*>(e + k0) = xv;
            if ((p & 7) == 0) bw[k0 >> 5] = word;
          }
        }
        return acc;
      };
      float acc;
      if constexpr (kFullPath) {
        acc = full_tile ? body(std::true_type{}, std::true_type{})
                        : body(std::true_type{}, std::false_type{});
      } else {
        acc = uni ? body(std::true_type{}, std::false_type{})
                  : body(std::false_type{}, std::false_type{});
      }
      if constexpr (kLate) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);  // the stage has been read
      }
      acc = warp_butterfly_sum(acc);
      if (lane == 0) ws[w][warp] = acc;
    }

    if ((uint32_t)p < nwn) s_sc[(ti + 1) & 1][p] = sc_next;
    if constexpr (LAMB) {
      if (p == 0 && VTn < n_vt) {
        cp_async_wait_all();
        LMeta& nx = s_lm[(ti + 1) & 1];
        nx.l = s_lr.l;
        nx.lend = s_lr.lend;
        nx.s = s_lr.s;
        nx.r = A.ratio_ef ? __fdiv_rn(s_lr.c2, s_lr.c1) : 1.0f;
      }
    }
    // one barrier per tile: the warp totals are double-buffered by parity
    // (the next tile writes the other half), and it also agrees on stopping
    const bool stop = named_sync_or(1, kConsumers, s_abort != 0);
    if ((uint32_t)p < wend - wbeg)
      A.ws.wpart[((uint64_t)(wbeg + p) * G.nc + tl.g) * G.tpc + tl.t] = tree8(ws[wbeg + p]);
    if (stop) break;
  }
}

template <bool BF16, bool LAMB, bool MSIGN>
cudaError_t run_compress(const CompressArgs& a, int sms, cudaStream_t s) {
  using S = CompressSmem<BF16, MSIGN>;
  static PerDeviceOnce once;
  const cudaError_t attr = once.run([] {
    return cudaFuncSetAttribute(k_compress<BF16, LAMB, MSIGN>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S::kBytes);
  });
  if (attr != cudaSuccess) return attr;
  const int grid =
      grid_for(k_compress<BF16, LAMB, MSIGN>, sms, a.geo.n_tiles, kCompressThreads, S::kBytes);
  k_compress<BF16, LAMB, MSIGN><<<grid, kCompressThreads, S::kBytes, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_compress(const CompressArgs& a, bool bf16, bool lamb, int sms,
                            cudaStream_t s) {
  if (bf16)
    return lamb ? run_compress<true, true, false>(a, sms, s)
                : run_compress<true, false, false>(a, sms, s);
  return lamb ? run_compress<false, true, false>(a, sms, s)
              : run_compress<false, false, false>(a, sms, s);
}

cudaError_t launch_compress_signm(const CompressArgs& a, bool bf16, bool lamb, int sms,
                                  cudaStream_t s) {
  if (bf16)
    return lamb ? run_compress<true, true, true>(a, sms, s)
                : run_compress<true, false, true>(a, sms, s);
  return lamb ? run_compress<false, true, true>(a, sms, s)
              : run_compress<false, false, true>(a, sms, s);
}

}  // namespace ob
