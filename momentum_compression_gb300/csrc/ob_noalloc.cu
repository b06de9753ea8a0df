// ob_compress_noalloc: the worker compression of ob_compress (1-bit Adam)
// for callers that cannot allocate device memory, and
// ob_noalloc_device_error, which reads its device error word.
//
// Who needs it: code that lives inside a host runtime which owns the
// device's memory through its own pool and hands its extensions no
// allocator (a cudaMalloc behind the pool's back can fail once the pool has
// reserved the device, and breaks the pool's accounting), and code on a
// path where the implicit device-wide synchronisation of cudaMalloc and
// cudaFree is not acceptable.  Such callers can still own the inputs and
// outputs, but not the scratch area ob_set_workspace() asks for.
//
// This entry point therefore takes its scratch from the file-scope array
// g_scratch below, which every GPU that loads the library holds until the
// process exits:
//   [0, kScratchBytes - 256)              per-(worker, chunk, tile) totals
//                                         of |x|, written before they are read
//                                         by every call
//   [kScratchBytes - 256, +4)             the device error word
// Host code cannot use the array's name as a device address: the first call
// on each device (of either entry point) looks the address up with
// cudaGetSymbolAddress, with that device current, keeps it, and clears the
// error word once.  That first call should therefore come before any stream
// capture.  Every call shares the one array, so calls that overlap on the
// GPU (different streams, or different host threads on one device) race.
//
// The error word is sticky: a bounded wait that gives up records its code
// only if the word holds 0, no call clears it, and ob_noalloc_device_error
// returns it and clears it.  A failure therefore stays visible until it has
// been read, however many calls follow.
#include <cstdio>
#include <mutex>

#include "ob_internal.cuh"

namespace {

constexpr size_t kScratchBytes = OB_NOALLOC_SCRATCH_BYTES;
constexpr size_t kErrOffset = kScratchBytes - 256;  // the error word's byte offset
static_assert(kScratchBytes % 256 == 0, "the scratch size must be a multiple of 256 bytes");
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The current device's address of g_scratch, looked up (and its error word
// cleared on `s`) on the first call for that device.
cudaError_t scratch_base(void** base, cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(static_cast<char*>(p) + kErrOffset, 0, sizeof(unsigned), s);
    if (e != cudaSuccess) return e;
    g_addr[dev] = p;
  }
  *base = g_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" ob_status ob_compress_noalloc(ob_ctx* ctx, const void* const* grads,
                                         const float* m, float* const* err, uint32_t* bits,
                                         float* scales, ob_stream_t stream) {
  OB_TRACE();
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
  // W * n_chunks * tiles_per_chunk totals of 4 bytes must fit below the
  // error word: the exact rule ob.h states.
  const size_t part_bytes = (size_t)G.W * G.nc * G.tpc * sizeof(float);
  if (part_bytes > kErrOffset) {
    char msg[256];
    snprintf(msg, sizeof msg,
             "compress_noalloc: this layout needs %zu bytes of per-tile totals, the static "
             "scratch holds %zu (use ob_compress with a workspace)",
             part_bytes, kErrOffset);
    return ob::ctx_fail(ctx, OB_ERR_UNSUPPORTED, msg);
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  void* base = nullptr;
  if (e == cudaSuccess) e = scratch_base(&base, s);
  if (e != cudaSuccess) return ob::ctx_fail(ctx, OB_ERR_CUDA, cudaGetErrorString(e));

  ob::CompressArgs a{};
  a.geo = G;
  a.nw = G.W;
  a.ws.wpart = static_cast<float*>(base);
  a.ws.err = reinterpret_cast<unsigned*>(static_cast<char*>(base) + kErrOffset);
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
  if (e == cudaSuccess) e = ob::launch_finalize_scales(G, a.ws.wpart, G.W, scales, sms, s);
  if (e != cudaSuccess) return ob::ctx_fail(ctx, OB_ERR_CUDA, cudaGetErrorString(e));
  return OB_OK;
}

extern "C" ob_status ob_noalloc_device_error(unsigned* code, ob_stream_t stream) {
  OB_TRACE();
  if (!code) return ob::ctx_fail(nullptr, OB_ERR_INVALID, "noalloc_device_error: code is NULL");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  void* base = nullptr;
  unsigned v = 0;
  cudaError_t e = scratch_base(&base, s);
  if (e == cudaSuccess) {
    unsigned* word = reinterpret_cast<unsigned*>(static_cast<char*>(base) + kErrOffset);
    e = cudaMemcpyAsync(&v, word, sizeof v, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(word, 0, sizeof v, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  }
  if (e != cudaSuccess) return ob::ctx_fail(nullptr, OB_ERR_CUDA, cudaGetErrorString(e));
  *code = v;
  return OB_OK;
}
