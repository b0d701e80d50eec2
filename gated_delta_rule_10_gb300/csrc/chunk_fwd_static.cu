// gdr_chunk_fwd_static: the chunked forward for callers that cannot allocate
// device memory when they call the library.
//
// Some callers are not allowed to call cudaMalloc at the moment they run the
// forward pass: a plugin whose host framework owns every device allocation
// and forbids new ones while it enqueues work, or a latency-critical loop in
// which cudaMalloc may block or implicitly synchronise the device. Such a
// caller cannot provide the small workspace gdr_chunk_fwd asks for. This entry
// point uses a fixed scratch area compiled into the library instead: a
// file-scope __device__ array that every GPU using the library holds from the
// moment the library's code is loaded on it until the process exits.
//
// The scratch only holds the status words of the tensor-core kernels (a
// device-side wait that gave up records itself there). Its size is fixed at
// kStaticScratchBytes; a request that needs more scratch is rejected with
// GDR_ERR_WORKSPACE before anything is enqueued.
//
// Sharing: all calls on a device use the same array, and it keeps whatever the
// last call left in it. Each call clears the status words on its stream before
// its kernel runs. Calls whose work overlaps on the GPU (for instance on two
// streams without ordering between them) race on the status words; order such
// calls on one stream. gdr_chunk_fwd_static_check reads the status words the
// last call on a device left there (the report of a device-side wait that gave
// up), once that call's work has finished.
//
// Set-up: the first call on each device looks up the array's device address
// (cudaGetSymbolAddress, with that device current) and caches it. Make that
// first call before any stream capture begins. `stream` must belong to the
// current device (a stream of another device is rejected). A lookup that
// fails clears the cached address, so a call after cudaDeviceReset looks it
// up again.
#include <mutex>

#include "gdr.h"
#include "kernels.h"

namespace {

constexpr size_t kStaticScratchBytes = 256;
constexpr int kMaxDevices = 64;
// the scratch holds the minimum workspace, which is the status words alone
static_assert(kStaticScratchBytes >= gdr::kChunkWorkspaceBytes, "minimum workspace fits");
static_assert(gdr::kStatusWords * sizeof(int) <= kStaticScratchBytes, "status words fit");

static __device__ __align__(256) unsigned char g_scratch[kStaticScratchBytes];

std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// The current device, checked against the device that owns `stream`.
gdr_status current_device(gdr_stream_t stream, int* dev) {
  if (cudaGetDevice(dev) != cudaSuccess || *dev < 0) return GDR_ERR_CUDA;
  if (*dev >= kMaxDevices) return GDR_ERR_UNSUPPORTED;
  if (stream) {
    int sdev = -1;
    if (cudaStreamGetDevice(reinterpret_cast<cudaStream_t>(stream), &sdev) != cudaSuccess)
      return GDR_ERR_INVALID_ARG;
    if (sdev != *dev) return GDR_ERR_INVALID_ARG;
  }
  return GDR_OK;
}

// Device address of g_scratch on device `dev`, the current one (looked up once
// per device; a failed lookup clears the cache entry).
gdr_status scratch_address(int dev, void** out) {
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) {
      g_scratch_addr[dev] = nullptr;
      return GDR_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return GDR_OK;
}

}  // namespace

extern "C" gdr_status gdr_chunk_fwd_static(const gdr_shape* shape, const void* q, const void* k,
                                           const void* v, const float* g, const float* beta,
                                           const float* lam, const void* b, const void* w,
                                           const float* h0, void* o, float* hT,
                                           gdr_stream_t stream) {
  size_t need = 0;
  const gdr_status st = gdr_chunk_fwd_workspace_min(shape, &need);
  if (st != GDR_OK) return st;
  if (need > kStaticScratchBytes) return GDR_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (need > 0) {
    int dev = -1;
    gdr_status sa = current_device(stream, &dev);
    if (sa == GDR_OK) sa = scratch_address(dev, &scratch);
    if (sa != GDR_OK) return sa;
  }
  const gdr_status rc = gdr_chunk_fwd(shape, q, k, v, g, beta, lam, b, w, h0, o, hT, scratch,
                                      need > 0 ? kStaticScratchBytes : 0, stream);
  if (rc == GDR_ERR_CUDA && need > 0) {   // e.g. after cudaDeviceReset: look it up again
    int dev = -1;
    if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < kMaxDevices) {
      std::lock_guard<std::mutex> lock(g_mutex);
      g_scratch_addr[dev] = nullptr;
    }
  }
  return rc;
}

extern "C" gdr_status gdr_chunk_fwd_static_check(gdr_stream_t stream, int* detail) {
  int dev = -1;
  gdr_status sa = current_device(stream, &dev);
  void* scratch = nullptr;
  if (sa == GDR_OK) sa = scratch_address(dev, &scratch);
  if (sa != GDR_OK) return sa;
  return gdr_chunk_fwd_check(scratch, stream, detail);
}
