// ob_compress_noalloc: the worker compression of ob_compress (1-bit Adam)
// for callers that cannot allocate device memory.
//
// Who needs it: code that lives inside a host runtime which owns the
// device's memory through its own pool and hands its extensions no
// allocator (a cudaMalloc behind the pool's back can fail once the pool has
// reserved the device, and breaks the pool's accounting), and code on a
// path where the implicit device-wide synchronisation of cudaMalloc and
// cudaFree is not acceptable.  Such callers can still own the inputs and
// outputs, but not the scratch area ob_set_workspace() asks for.
//
// This entry point therefore takes its scratch -- the per-(worker, tile)
// totals of |x| and a device error word -- from the file-scope array
// g_scratch below, which every GPU that loads the library holds until the
// process exits.  Host code cannot use the array's name as a device
// address: the first call on each device looks the address up with
// cudaGetSymbolAddress (with that device current) and keeps it.  That
// first call should therefore come before any stream capture.  Every call
// shares the one array and overwrites it, so calls that overlap on the GPU
// (different streams, or different host threads on one device) race; the
// error word is cleared at the start of each call, and the totals need no
// clearing (each call writes all it reads).
#include <cstdio>
#include <mutex>

#include "ob_internal.cuh"

namespace {

constexpr size_t kScratchBytes = OB_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" ob_status ob_compress_noalloc(ob_ctx* ctx, const void* const* grads,
                                         const float* m, float* const* err, uint32_t* bits,
                                         float* scales, ob_stream_t stream) {
  if (!ctx) return ob::ctx_fail(nullptr, OB_ERR_INVALID, "ctx is NULL");
  const ob::Geo& G = *ob::ctx_geo(ctx);
  const ob_config& cfg = *ob::ctx_config(ctx);
  if (!grads || !err || !m || !bits || !scales)
    return ob::ctx_fail(ctx, OB_ERR_INVALID, "compress_noalloc: a buffer is NULL");
  for (uint32_t w = 0; w < G.W; ++w) {
    if (!grads[w] || !err[w])
      return ob::ctx_fail(ctx, OB_ERR_INVALID, "compress_noalloc: a worker buffer is NULL");
    if (!aligned16(grads[w]) || !aligned16(err[w]))
      return ob::ctx_fail(ctx, OB_ERR_ALIGN,
                          "compress_noalloc: worker buffers must be 16-byte aligned");
  }
  if (!aligned16(m) || !aligned16(bits) || (reinterpret_cast<uintptr_t>(scales) & 3u))
    return ob::ctx_fail(ctx, OB_ERR_ALIGN,
                        "compress_noalloc: m and bits must be 16-byte aligned, scales 4-byte");
  const size_t part_bytes = ((size_t)G.W * G.nc * G.tpc * sizeof(float) + 255) / 256 * 256;
  if (part_bytes + 256 > kScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof msg,
             "compress_noalloc: this layout needs %zu bytes of scratch, the static scratch "
             "holds %zu (use ob_compress with a workspace)",
             part_bytes + 256, kScratchBytes);
    return ob::ctx_fail(ctx, OB_ERR_UNSUPPORTED, msg);
  }
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return ob::ctx_fail(ctx, OB_ERR_CUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return ob::ctx_fail(ctx, OB_ERR_UNSUPPORTED, "compress_noalloc: device index too large");
  void* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev]) {
      e = cudaGetSymbolAddress(&g_addr[dev], g_scratch);
      if (e != cudaSuccess) {
        g_addr[dev] = nullptr;
        return ob::ctx_fail(ctx, OB_ERR_CUDA, cudaGetErrorString(e));
      }
    }
    base = g_addr[dev];
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  float* part = static_cast<float*>(base);
  unsigned* errw = reinterpret_cast<unsigned*>(static_cast<char*>(base) + part_bytes);
  e = cudaMemsetAsync(errw, 0, sizeof(unsigned), s);
  if (e != cudaSuccess) return ob::ctx_fail(ctx, OB_ERR_CUDA, cudaGetErrorString(e));

  ob::CompressArgs a{};
  a.geo = G;
  a.ws.wpart = part;
  a.ws.err = errw;
  for (uint32_t w = 0; w < G.W; ++w) {
    a.g[w] = grads[w];
    a.e[w] = err[w];
  }
  a.m = m;
  a.bits = bits;
  a.scales = scales;
  a.ratio_ef = 1;
  a.b1 = cfg.b1;
  a.ob1 = 1.0f - cfg.b1;
  a.clip = cfg.clip_value;
  e = ob::launch_compress(a, cfg.grad_dtype == OB_GRAD_BF16, false, sms, s);
  if (e == cudaSuccess) e = ob::launch_finalize_scales(G, part, G.W, scales, sms, s);
  if (e != cudaSuccess) return ob::ctx_fail(ctx, OB_ERR_CUDA, cudaGetErrorString(e));
  return OB_OK;
}
