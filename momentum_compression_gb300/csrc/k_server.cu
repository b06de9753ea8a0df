// Server side of the 1-bit compressed optimizer step: every server j
// averages the W workers' compressed chunks of its partition, adds its own
// error and compresses again (1-bit LAMB summary, paragraphs 3-4: the
// server error delta~ and the 3-phase Alltoall/AllGather exchange).
//
// Per element k of chunk g:
//   z    = (sum over w = 0..W-1, in order, from 0, of scale_w(g)*sign_w(k)) / W
//   e_s  = y_prev - sscale_prev*sign(y_prev)   (deferred server error)
//   y    = rho_l*e_s + z                        (1-bit Adam: e_s + z)
//   sbit = y >= 0; y is stored in place of e_s
//   sscale(g) = mean |y| over the chunk: this kernel writes one total per
//   tile; k_finalize_scales adds them in tile order
//
// The workers' words are laid out worker-major with a 16-byte aligned row
// stride, so the W-way gather of one tile is W contiguous runs of 512
// bytes.  A producer thread streams, per tile, the e_s tile and the W runs
// (rounded out to 16-byte boundaries) into a ring of shared-memory stages
// with cp.async.bulk; eight consumer warps read the four words each lane
// needs from shared memory.  Waits are bounded (ptx.cuh).
//
// The W-way signed sum depends only on the element's W sign bits, and the
// scales are constant within a tile.  So each tile first tabulates
// z8[b] = (sum over w < min(W,8), in order, from 0, of (bit w of b ? s_w :
// -s_w)) for all 2^min(W,8) patterns b -- the same additions in the same
// order as element by element, hence the same bits -- divided by W when
// W <= 8.  An element then gathers its first 8 workers' bits into a byte
// (an 8 x 4 bit transpose of the lane's nibbles) and reads its z from the
// table; workers 8.. are added after it in order: for W = 16 one select and
// addition per element and worker, for any other W two elements at a time
// -- per tile, a table holds for each such worker w the four pairs
// (+-s_w, +-s_w) a lane's two sign bits select, and one paired addition
// (add.rn.f32x2, each half rounded as on its own) adds worker w's terms to
// two elements' sums.
#include <type_traits>

#include "ob_internal.cuh"
#include "ptx.cuh"

namespace ob {
namespace {

constexpr int kSConsumers = kThreads;
constexpr int kServerThreads = kThreads + 32;
constexpr uint32_t kRunWords = kTile / 32 + 8;  // one tile's words + rounding slack

// Per-tile scalars, written by the producer into each stage next to the
// copies (plain shared stores made visible by its release-arrive on the
// stage's mbarrier): the decoded tile, the previous server scale of its
// chunk and, for 1-bit LAMB, the tile's first layer, that layer's end and
// its rho.  The consumers take them from the stage and wait on nothing
// else at a tile start.
struct TileHdr {
  Tile tl;
  float osc, r;
  uint32_t l, pad;
  uint64_t lend;
};
constexpr size_t kHdrBytes = 64;
static_assert(sizeof(TileHdr) <= kHdrBytes && kHdrBytes % 16 == 0, "stage header");

// Stages in the ring: 3 up to 8 workers (3 CTAs per SM); beyond that a
// stage holds more word runs and the per-element sums are longer, and 2
// stages keep 3 CTAs per SM where 3 would allow only 2.
template <uint32_t WT>
__host__ __device__ constexpr int server_stages() {
  return WT != 0 && WT <= 8 ? 3 : 2;
}

struct ServerSmem {
  // the e_s tile, the W workers' word runs, the server's previous words
  // and the tile header
  __host__ __device__ static size_t hdr_offset(uint32_t W) {
    return kTile * 4 + (size_t)(W + 1) * kRunWords * 4;
  }
  __host__ __device__ static size_t stage_bytes(uint32_t W) { return hdr_offset(W) + kHdrBytes; }
  // the pair table of workers 8.. (two tiles' worth)
  __host__ __device__ static size_t pairs_bytes(uint32_t W) {
    return W > 8 && W != 16 ? 2 * (size_t)(W - 8) * 4 * 8 : 0;
  }
  __host__ __device__ static size_t bytes(uint32_t W, int stages) {
    return stages * stage_bytes(W) + (2 * stages) * 8 + 3 * OB_MAX_WORKERS * 4 + 2 * 256 * 4 +
           pairs_bytes(W);
  }
};

// Table entry b for the first W8 = min(W, 8) workers (see the file header).
// The division by W (W <= 8) is the exact multiply by 1/W when W is a
// power of two (inv_w != 0).
__device__ __forceinline__ float z8_entry(const float* sc, uint32_t W, float inv_w, uint32_t b) {
  const uint32_t W8 = W < 8 ? W : 8;
  float z = 0.0f;
  for (uint32_t w = 0; w < W8; ++w) z = __fadd_rn(z, ((b >> w) & 1u) ? sc[w] : -sc[w]);
  return W <= 8 ? div_by_workers(z, (float)W, inv_w) : z;
}

// WT: the worker count when it is a compile-time 4, 8 or 16 (the tables'
// and loops' bounds are then constants), 0 for any other W.
template <bool LAMB, uint32_t WT>
__global__ void __launch_bounds__(kServerThreads, 3) k_server(const ServerArgs A) {
  constexpr int kSStages = server_stages<WT>();
  extern __shared__ __align__(128) unsigned char smem[];
  const Geo& G = A.geo;
  const size_t stage_bytes = ServerSmem::stage_bytes(G.W);
  unsigned char* stage0 = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kSStages * stage_bytes);
  uint64_t* empty = full + kSStages;
  float(*s_sc)[OB_MAX_WORKERS] = reinterpret_cast<float(*)[OB_MAX_WORKERS]>(empty + kSStages);
  float(*s_z8)[256] = reinterpret_cast<float(*)[256]>(s_sc + 3);
  // [2][W - 8][4] pairs (see the file header); 8-byte aligned after s_z8
  unsigned long long* s_pairs = reinterpret_cast<unsigned long long*>(s_z8 + 2);
  __shared__ float ws[2][8];
  __shared__ volatile int s_abort;
  const size_t hdr_off = ServerSmem::hdr_offset(G.W);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  unsigned* err = A.ws.err;
  const float fW = (float)G.W, inv_w = inv_workers(G.W);

  if (tid == 0) {
    for (int s = 0; s < kSStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kSConsumers / 32);
    }
    s_abort = 0;
    fence_barrier_init();
  }
  __syncthreads();

  // ------------------------------------------------------------ producer
  if (warp == kSConsumers / 32) {
    if (lane != 0) return;
    uint32_t ti = 0;
    bool ok = true;
    // 1-bit LAMB: the layer of the tile, loaded a tile before the loads
    // that depend on it
    [[maybe_unused]] uint32_t l_cur =
        LAMB && A.T0 + blockIdx.x < A.T1 ? __ldg(A.ws.tile_layer + A.T0 + blockIdx.x) : 0u;
    for (uint32_t T = A.T0 + blockIdx.x; T < A.T1; T += gridDim.x, ++ti) {
      const Tile tl = decode_tile(G, T);
      const uint64_t lstart = tl.start - A.base;  // the tile's index in this call's buffers
      // the header's loads go out before the wait for a free stage
      const float osc = __ldcg(A.sscales_old + (tl.g - A.g0));
      [[maybe_unused]] uint32_t l = 0;
      [[maybe_unused]] uint64_t lend = 0;
      [[maybe_unused]] float c2 = 1.0f, c1 = 1.0f;
      if constexpr (LAMB) {
        l = l_cur;
        lend = __ldg(A.ws.layer_off + l + 1);
        if (A.ratio_ef) {
          c2 = __ldg(A.c_prev2 + l);
          c1 = __ldg(A.c_prev + l);
        }
        if (T + gridDim.x < A.T1) l_cur = __ldg(A.ws.tile_layer + T + gridDim.x);
      }
      const uint32_t s = ti % kSStages, r = ti / kSStages;
      if (r >= 1) ok = mbar_wait(&empty[s], (r - 1) & 1, err, kErrWaitEmpty);
      if (!ok || s_abort) {
        ok = false;
        break;
      }
      const uint64_t w0 = (lstart >> 5) & ~uint64_t(3);
      const uint64_t w1 = ((lstart + tl.len) / 32 + 3) & ~uint64_t(3);
      const uint32_t run = (uint32_t)(w1 - w0) * 4;
      unsigned char* st = stage0 + s * stage_bytes;
      TileHdr* hd = reinterpret_cast<TileHdr*>(st + hdr_off);
      hd->tl = tl;
      hd->osc = osc;
      if constexpr (LAMB) {
        hd->l = l;
        hd->lend = lend;
        hd->r = A.ratio_ef ? __fdiv_rn(c2, c1) : 1.0f;
      }
      mbar_arrive_expect_tx(&full[s], tl.len * 4 + (G.W + 1) * run);
      bulk_g2s(st, A.e_s + lstart, tl.len * 4, &full[s]);
      for (uint32_t w = 0; w < G.W; ++w)
        bulk_g2s(st + kTile * 4 + (size_t)w * kRunWords * 4, A.bits + w * A.bits_stride + w0,
                 run, &full[s]);
      // the previous server words of this tile (only this CTA rewrites
      // them, after this copy has landed; the rounding words read beyond
      // the tile are not used).  They come from sbits_old, which is sbits
      // itself unless the caller double-buffers the server output.
      bulk_g2s(st + kTile * 4 + (size_t)G.W * kRunWords * 4, A.sbits_old + w0, run, &full[s]);
    }
    if (!ok) s_abort = 1;
    for (uint32_t k = 0; k < kSStages && k < ti; ++k) {
      const uint32_t t = ti - 1 - k;
      if (!mbar_wait(&full[t % kSStages], (t / kSStages) & 1, err, kErrDrain)) break;
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  const int p = tid;
  // the byte of a sign word holding this lane's nibble (selector for
  // byte_perm: that byte of the first and of the second operand) and the
  // nibble's offset in it
  const uint32_t bsel = ((p & 7) >> 1) | ((4 + ((p & 7) >> 1)) << 4);
  const uint32_t hs = 4 * (p & 1);
  const uint32_t Wc = WT ? WT : G.W;
  // scales of the first tile
  const uint32_t W8 = Wc < 8 ? Wc : 8;
  // the layer factor rho = c_prev2/c_prev of layer l (1 without the
  // step-ratio error feedback)
  auto rho = [&](uint32_t l) {
    return A.ratio_ef ? __fdiv_rn(__ldg(A.c_prev2 + l), __ldg(A.c_prev + l)) : 1.0f;
  };
  // One barrier per tile: the worker scales are loaded two tiles ahead
  // (ring of 3), so that the z table of tile t+1 can be built during tile
  // t from scales published by the barrier ending tile t-1; the tile
  // totals are double-buffered.
  // worker w's scale of chunk g
  auto wscale = [&](uint32_t w, uint32_t g) {
    return __ldcg(A.scales + (uint64_t)w * A.sc_stride + (g - A.g0));
  };
  if (A.T0 + blockIdx.x + gridDim.x < A.T1 && (uint32_t)p < Wc)
    s_sc[1][p] = wscale(p, decode_tile(G, A.T0 + blockIdx.x + gridDim.x).g);
  if (A.T0 + blockIdx.x < A.T1 && (uint32_t)p < Wc)
    s_sc[0][p] = wscale(p, decode_tile(G, A.T0 + blockIdx.x).g);
  named_sync(1, kSConsumers);
  if ((uint32_t)p < (1u << W8)) s_z8[0][p] = z8_entry(s_sc[0], Wc, inv_w, p);
  // entry b of worker w's pairs: (bit 0 of b ? s_w : -s_w, bit 1 of b ? s_w : -s_w)
  auto pairs_entry = [&](const float* sc, int q) {
    const uint32_t w = 8 + (uint32_t)q / 4, b = (uint32_t)q & 3u;
    const float sw = sc[w];
    return f2_make((b & 1u) ? sw : -sw, (b & 2u) ? sw : -sw);
  };
  const int n_pairs = WT == 0 && Wc > 8 ? (int)(Wc - 8) * 4 : 0;
  for (int q = p; q < n_pairs; q += kSConsumers) s_pairs[q] = pairs_entry(s_sc[0], q);
  named_sync(1, kSConsumers);
  uint32_t ti = 0;
  for (uint32_t T = A.T0 + blockIdx.x; T < A.T1; T += gridDim.x, ++ti) {
    const uint32_t s = ti % kSStages;
    // the worker scales of the tile after next
    float next_sc = 0.0f;
    const uint32_t Tn = T + gridDim.x, Tnn = Tn + gridDim.x;
    if (Tnn < A.T1 && (uint32_t)p < Wc) next_sc = wscale(p, decode_tile(G, Tnn).g);
    bool ok = s_abort == 0 && mbar_wait(&full[s], (ti / kSStages) & 1, err, kErrWaitFull);
    if (!ok) s_abort = 1;
    const unsigned char* st = stage0 + s * stage_bytes;
    // the tile's scalars from the stage header (after a failed wait the
    // tile is decoded here, so that addresses stay valid; the values are
    // discarded when the loop exits at the tile's end)
    const TileHdr& hd = *reinterpret_cast<const TileHdr*>(st + hdr_off);
    const Tile tl = ok ? hd.tl : decode_tile(G, T);
    const float osc = hd.osc;
    bool valid[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) valid[i] = 1024u * i + 4u * p < tl.len;
    const uint32_t* sbw = reinterpret_cast<const uint32_t*>(st + kTile * 4);
    const uint32_t* sow = sbw + Wc * kRunWords;  // the server's previous words
    const uint32_t wshift = (uint32_t)(((tl.start - A.base) >> 5) & 3);  // rounding of the runs

    const float* z8 = s_z8[ti & 1];
    [[maybe_unused]] const float* sc = s_sc[ti % 3];
    const unsigned long long* pairs = s_pairs + (ti & 1) * n_pairs;

    uint32_t l_t = 0;
    uint64_t lend_t = 0;
    float r_t = 1.0f;
    if constexpr (LAMB) {
      l_t = ok ? hd.l : 0u;
      lend_t = ok ? hd.lend : 0u;
      r_t = hd.r;
    }
    // FULL: all 4096 elements of the tile are real (no length or padding
    // checks per element).  UNI: the whole tile lies in one layer (rho
    // scalar); else the layers are walked element by element.
    auto work = [&](auto full_tag, auto uni_tag) -> float {
      constexpr bool FULL = decltype(full_tag)::value;
      [[maybe_unused]] constexpr bool UNI = decltype(uni_tag)::value;
      float4 ev[4];
      float z[4][4];
      uint32_t owd[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t off = 1024u * i + 4u * p;
        const bool vi = FULL || valid[i];
        ev[i] = vi ? *reinterpret_cast<const float4*>(st + off * 4)
                   : make_float4(0.f, 0.f, 0.f, 0.f);
        owd[i] = vi ? sow[(off >> 5) + wshift] : 0u;
#pragma unroll
        for (int c = 0; c < 4; ++c) z[i][c] = 0.0f;
        if (vi) {
          const uint32_t widx = (off >> 5) + wshift;
          const int sh = 4 * (p & 7);
          // byte c of idx = the first W8 workers' bits of element c: an
          // 8 x 4 bit transpose.  Gather the byte holding this lane's nibble
          // from each word (workers 0-3 in xa, 4-7 in xb, absent workers
          // 0), keep the nibbles (idx byte w: worker w's 4 bits low, worker
          // w+4's high), then two delta swaps transpose the two 4 x 4 bit
          // blocks (the 2 x 2 sub-blocks, then the bits inside them).
          uint32_t wv[8];
#pragma unroll
          for (uint32_t w = 0; w < 8; ++w) wv[w] = w < W8 ? sbw[w * kRunWords + widx] : 0u;
          const uint32_t xa = __byte_perm(__byte_perm(wv[0], wv[1], bsel),
                                          __byte_perm(wv[2], wv[3], bsel), 0x5410);
          const uint32_t xb = __byte_perm(__byte_perm(wv[4], wv[5], bsel),
                                          __byte_perm(wv[6], wv[7], bsel), 0x5410);
          uint32_t idx = ((xa >> hs) & 0x0F0F0F0Fu) | ((xb << (4 - hs)) & 0xF0F0F0F0u);
          uint32_t tsw = ((idx >> 14) ^ idx) & 0x0000CCCCu;
          idx ^= tsw ^ (tsw << 14);
          tsw = ((idx >> 7) ^ idx) & 0x00AA00AAu;
          idx ^= tsw ^ (tsw << 7);
#pragma unroll
          for (int c = 0; c < 4; ++c) z[i][c] = z8[__byte_perm(idx, 0u, 0x4440u | c)];
          if (WT > 8) {
            // a compile-time 16: the worker loop unrolled, one select and
            // one addition per element and worker (on the integer and FP
            // pipes; the pair table's loads measured slower here)
#pragma unroll
            for (uint32_t w = 8; w < Wc; ++w) {
              const uint32_t wd = sbw[w * kRunWords + widx] >> sh;
              const float scw = sc[w];
#pragma unroll
              for (int c = 0; c < 4; ++c)
                z[i][c] = __fadd_rn(z[i][c], ((wd >> c) & 1u) ? scw : -scw);
            }
          } else if (WT == 0) {
            unsigned long long z01 = f2_make(z[i][0], z[i][1]);
            unsigned long long z23 = f2_make(z[i][2], z[i][3]);
#pragma unroll 8
            for (uint32_t w = 8; w < Wc; ++w) {
              const uint32_t wd = sbw[w * kRunWords + widx] >> sh;
              const unsigned long long* pw = pairs + (w - 8) * 4;
              z01 = f2_add(z01, pw[wd & 3u]);
              z23 = f2_add(z23, pw[(wd >> 2) & 3u]);
            }
            f2_split(z01, z[i][0], z[i][1]);
            f2_split(z23, z[i][2], z[i][3]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);

      float acc = 0.0f;
      [[maybe_unused]] uint32_t l = l_t;
      [[maybe_unused]] uint64_t lend = lend_t;
      [[maybe_unused]] float r_l = r_t;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint64_t k0 = tl.start + 1024u * i + 4u * p;
        float4 yv;
        uint32_t nib = 0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint64_t k = k0 + c;
          float y = 0.0f;
          if (FULL || (valid[i] && k < G.n)) {
            const float zc = Wc <= 8 ? z[i][c] : div_by_workers(z[i][c], fW, inv_w);
            const float so = signed_by_bit(osc, owd[i] >> (4 * (p & 7)), c);
            const float et = __fsub_rn(f4get(ev[i], c), so);
            if constexpr (LAMB) {
              if constexpr (!UNI) {
                if (advance_layer(A.ws.layer_off, G.L, k, l, lend)) r_l = rho(l);
              }
              y = __fadd_rn(__fmul_rn(r_l, et), zc);
            } else {
              y = __fadd_rn(et, zc);
            }
            acc = __fadd_rn(acc, fabsf(y));
            if (y >= 0.0f) nib |= 1u << c;
          }
          f4at(yv, c) = y;
        }
        const uint32_t word = pack_word(nib, lane);
        if (FULL || valid[i]) {
          *reinterpret_cast<float4*>(A.e_s + (k0 - A.base)) = yv;
          if ((p & 7) == 0) A.sbits[(k0 - A.base) >> 5] = word;
        }
      }
      return acc;
    };
    const bool full_tile = tl.len == kTile && tl.start + kTile <= G.n;
    const bool uni = !LAMB || tl.start + tl.len <= lend_t || G.n <= lend_t;
    float acc;
    if (full_tile) {
      if (!LAMB || uni) acc = work(std::true_type{}, std::true_type{});
      else acc = work(std::true_type{}, std::false_type{});
    } else {
      if (!LAMB || uni) acc = work(std::false_type{}, std::true_type{});
      else acc = work(std::false_type{}, std::false_type{});
    }
    acc = warp_butterfly_sum(acc);
    if (lane == 0) ws[ti & 1][warp] = acc;
    if (Tnn < A.T1 && (uint32_t)p < Wc) s_sc[(ti + 2) % 3][p] = next_sc;
    if (Tn < A.T1) {
      if ((uint32_t)p < (1u << W8))
        s_z8[(ti + 1) & 1][p] = z8_entry(s_sc[(ti + 1) % 3], Wc, inv_w, p);
      for (int q = p; q < n_pairs; q += kSConsumers)
        s_pairs[((ti + 1) & 1) * n_pairs + q] = pairs_entry(s_sc[(ti + 1) % 3], q);
    }
    const bool stop = named_sync_or(1, kSConsumers, s_abort != 0);
    if (p == 0) A.ws.spart[(uint64_t)tl.g * G.tpc + tl.t] = tree8(ws[ti & 1]);
    if (stop) break;
  }
}

template <bool LAMB, uint32_t WT>
cudaError_t run_server(const ServerArgs& a, int sms, cudaStream_t s) {
  constexpr int kSt = server_stages<WT>();
  const size_t bytes = ServerSmem::bytes(a.geo.W, kSt);
  static PerDeviceOnce once;
  const cudaError_t attr = once.run([] {
    return cudaFuncSetAttribute(k_server<LAMB, WT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)ServerSmem::bytes(WT ? WT : OB_MAX_WORKERS, kSt));
  });
  if (attr != cudaSuccess) return attr;
  const int grid = grid_for(k_server<LAMB, WT>, sms, a.T1 - a.T0, kServerThreads, bytes);
  k_server<LAMB, WT><<<grid, kServerThreads, bytes, s>>>(a);
  return cudaGetLastError();
}

template <bool LAMB>
cudaError_t run_server_w(const ServerArgs& a, int sms, cudaStream_t s) {
  if (a.geo.W == 8) return run_server<LAMB, 8>(a, sms, s);
  if (a.geo.W == 4) return run_server<LAMB, 4>(a, sms, s);
  if (a.geo.W == 16) return run_server<LAMB, 16>(a, sms, s);
  return run_server<LAMB, 0>(a, sms, s);
}

}  // namespace

cudaError_t launch_server(const ServerArgs& a, bool lamb, int sms, cudaStream_t s) {
  return lamb ? run_server_w<true>(a, sms, s) : run_server_w<false>(a, sms, s);
}

}  // namespace ob
