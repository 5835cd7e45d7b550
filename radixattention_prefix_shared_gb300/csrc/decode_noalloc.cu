// sgl_decode_attention_noalloc: decode attention for callers that cannot
// allocate device memory.
//
// Some callers of this library are not allowed to call cudaMalloc (or any
// allocating routine) when they run attention: runtimes whose memory planner
// fixes every device buffer at start-up and forbids allocation afterwards,
// and plugin-style hosts that hand a kernel only its input and output
// buffers.  sgl_decode_attention needs a caller-provided scratch buffer for
// its split-KV partial results; this entry point takes its scratch from a
// fixed array in the library's own device memory instead.
//
// The array is a file-scope static __device__ buffer of kScratchBytes; every
// GPU that loads this module holds it until the process exits.  Host code
// cannot use the array's name as a device address, so the device address is
// looked up with cudaGetSymbolAddress once per device and CUDA context (on
// the first call made with that device current in that context) and cached.
// Each context loads the module at its own address, so a caller that makes
// its own driver-API context gets that context's copy of the array.  A device
// reset after the first call is not supported: the module is loaded again
// at an address this cache does not know.  All calls share the array: calls
// whose kernels overlap on the GPU (different streams, or different host
// threads without ordering) race on it and must be serialised by the caller.
// The scheduling kernel rewrites every part of the scratch that is read
// later, so nothing needs clearing between calls.
#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace sgl {
namespace {

constexpr size_t kScratchBytes = (size_t)SGL_DECODE_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) uint8_t g_decode_scratch[kScratchBytes];

// (device, context) -> the array's device address there
struct ScratchEntry {
  int dev;
  void* ctx;
  void* ptr;
};
constexpr int kMaxEntries = 64;
std::mutex g_scratch_mu;
ScratchEntry g_scratch[kMaxEntries] = {};
int g_scratch_n = 0;

// The current context (cuCtxGetCurrent, reached through the runtime so that
// the library needs no link against the driver library), or nullptr.
void* current_context() {
  using Fn = CUresult (*)(CUcontext*);
  static Fn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<Fn>(f);
  }();
  CUcontext c = nullptr;
  if (fn == nullptr || fn(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

// Device address of g_decode_scratch on the current device and context
// (looked up once per pair).
sgl_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SGL_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  auto cached = [&](void* ctx) -> void* {
    for (int i = 0; i < g_scratch_n; ++i)
      if (g_scratch[i].dev == dev && g_scratch[i].ctx == ctx) return g_scratch[i].ptr;
    return nullptr;
  };
  void* ctx = current_context();
  if (ctx != nullptr) {
    if (void* p = cached(ctx)) {
      *out = p;
      return SGL_OK;
    }
  }
  // first call in this context (the lookup also makes the device's primary
  // context current when the thread has none yet)
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return SGL_ERR_CUDA;
  if (ctx == nullptr) ctx = current_context();
  if (ctx != nullptr && cached(ctx) == nullptr) {
    if (g_scratch_n == kMaxEntries) return SGL_ERR_UNSUPPORTED;
    g_scratch[g_scratch_n++] = {dev, ctx, p};
  }
  *out = p;
  return SGL_OK;
}

}  // namespace
}  // namespace sgl

extern "C" sgl_status sgl_decode_attention_noalloc(
    const void* q, const void* pool_k, const void* pool_v, const int32_t* req_to_token,
    int32_t rtt_rows, int32_t rtt_stride, const int32_t* req_pool_idx, const int32_t* seq_lens,
    int32_t batch, int32_t max_seq_len, void* out, const sgl_attn_dims* dims,
    sgl_stream_t stream) {
  // the same checks, in the same order, as sgl_decode_attention makes before
  // it looks at its workspace
  float scale = 0.f;
  const sgl_status ok = sgl::validate_decode_call(q, pool_k, pool_v, req_to_token, rtt_rows, rtt_stride,
                                                  req_pool_idx, seq_lens, batch, max_seq_len, out, dims,
                                                  &scale);
  if (ok != SGL_OK || batch == 0) return ok;
  // reject, on the host and before any device call, work whose split-KV
  // scratch would not fit in the fixed array
  const size_t need = sgl_decode_workspace_bytes(batch, max_seq_len, dims);
  if (need == 0 || need > sgl::kScratchBytes) return SGL_ERR_WORKSPACE;
  void* scratch = nullptr;
  const sgl_status st = sgl::scratch_address(&scratch);
  if (st != SGL_OK) return st;
  return sgl_decode_attention(q, pool_k, pool_v, req_to_token, rtt_rows, rtt_stride, req_pool_idx,
                              seq_lens, batch, max_seq_len, out, scratch, sgl::kScratchBytes, dims,
                              stream);
}
