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
// looked up with cudaGetSymbolAddress once per device (on the first call on
// that device, with that device current) and cached.  All calls share the
// array: calls whose kernels overlap on the GPU (different streams, or
// different host threads without ordering) race on it and must be serialised
// by the caller.  The scheduling kernel rewrites every part of the scratch
// that is read later, so nothing needs clearing between calls.
#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace sgl {
namespace {

constexpr size_t kScratchBytes = (size_t)SGL_DECODE_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) uint8_t g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device (looked up once).
sgl_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SGL_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SGL_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr)
      return SGL_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return SGL_OK;
}

}  // namespace
}  // namespace sgl

extern "C" sgl_status sgl_decode_attention_noalloc(
    const void* q, const void* pool_k, const void* pool_v, const int32_t* req_to_token,
    int32_t rtt_rows, int32_t rtt_stride, const int32_t* req_pool_idx, const int32_t* seq_lens,
    int32_t batch, int32_t max_seq_len, void* out, const sgl_attn_dims* dims,
    sgl_stream_t stream) {
  if (dims == nullptr || dims->num_q_heads <= 0 || dims->num_kv_heads <= 0)
    return SGL_ERR_INVALID_ARG;
  if (batch < 0 || max_seq_len < 0) return SGL_ERR_INVALID_ARG;
  if (batch == 0) return SGL_OK;
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
