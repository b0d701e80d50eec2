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
// calls on one stream. A status recorded here is not returned to the caller;
// use gdr_chunk_fwd with a workspace and gdr_chunk_fwd_check when that report
// is needed.
//
// Set-up: the first call on each device looks up the array's device address
// (cudaGetSymbolAddress, with that device current) and caches it. Make that
// first call before any stream capture begins.
#include <mutex>

#include "gdr.h"
#include "kernels.h"

namespace {

constexpr size_t kStaticScratchBytes = 256;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_scratch[kStaticScratchBytes];

std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_scratch on the current device (looked up once per device).
gdr_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return GDR_ERR_CUDA;
  if (dev >= kMaxDevices) return GDR_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return GDR_ERR_CUDA;
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
    const gdr_status sa = scratch_address(&scratch);
    if (sa != GDR_OK) return sa;
  }
  return gdr_chunk_fwd(shape, q, k, v, g, beta, lam, b, w, h0, o, hT, scratch,
                       need > 0 ? kStaticScratchBytes : 0, stream);
}
