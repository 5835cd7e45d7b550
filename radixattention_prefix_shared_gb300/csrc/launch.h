// Host-side launchers (one per kernel family) and device queries.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>
#include <utility>

#include "../../include/sgl_attn.h"

namespace sgl {

// SM count of the current device (cached per device).
int num_sms();

// Limit of the extend and cascade-group kernels' bounded waits on their
// stage barriers, for launches made from now on (sgl_set_device_wait_limit_ns).
uint64_t device_wait_limit_ns();

// Raises kernel Kern's dynamic shared memory limit to `smem` bytes and returns
// how many of its blocks of `threads` fit on one SM (>= 1), or -1 on a CUDA
// error.  Done once per device and kernel: later calls (including calls made
// while a stream is being captured into a CUDA graph) only read the cache.
template <auto Kern>
int kernel_blocks_per_sm(int smem, int threads) {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  const bool cached = dev >= 0 && dev < 64;
  if (cached) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  if (cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return -1;
  int b = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, Kern, threads, (size_t)smem) != cudaSuccess)
    return -1;
  if (b < 1) b = 1;
  if (cached) cache[dev].store(b, std::memory_order_relaxed);
  return b;
}

sgl_status launch_store_kv(const void* k_new, const void* v_new, const int32_t* slots, int32_t n,
                           void* pool_k, void* pool_v, int32_t row_bytes, cudaStream_t stream);
// bf16 rows of row_elems values quantised into e4m3 pool rows
sgl_status launch_store_kv_fp8(const void* k_new, const void* v_new, const int32_t* slots,
                               int32_t n, void* pool_k, void* pool_v, int32_t row_elems,
                               float k_scale, float v_scale, cudaStream_t stream);

struct DecodeArgs {
  const void* q;
  const void* pool_k;
  const void* pool_v;
  const int32_t* req_to_token;
  int32_t rtt_stride;
  const int32_t* req_pool_idx;
  const int32_t* seq_lens;
  int32_t batch, max_seq_len;
  void* out;
  void* workspace;
  size_t workspace_bytes;
  int32_t num_q_heads, num_kv_heads, head_dim;
  float sm_scale;
  // cascade decode: shared-prefix groups (cascade == false: plain decode,
  // the fields below are unused)
  bool cascade = false;
  const int32_t* group_start = nullptr;
  const int32_t* group_len = nullptr;
  const int32_t* group_depth = nullptr;
  const int32_t* group_member_off = nullptr;
  const int32_t* group_members = nullptr;
  int32_t n_groups = 0, max_group_members = 0, max_depth = 0;
  // e4m3 pool (kv_fp8): pool rows hold codes; K/V values are code * scale
  bool kv_fp8 = false;
  float k_scale = 1.f, v_scale = 1.f;
};
// bytes in front of a cascade workspace: word 0 is the bounded-wait status
constexpr size_t kCascadeStatusBytes = 256;
size_t decode_workspace_bytes(int32_t batch, int32_t max_seq_len, int32_t num_q_heads,
                              int32_t num_kv_heads, int32_t head_dim, bool cascade = false,
                              int32_t max_depth = 0);
sgl_status launch_decode(const DecodeArgs& a, cudaStream_t stream);
// SGL_OK when the decode kernels are built for Hq query heads over Hkv KV
// heads (Hq % Hkv == 0 checked by the caller), else SGL_ERR_UNSUPPORTED.
sgl_status decode_shape_supported(int32_t num_q_heads, int32_t num_kv_heads);
// The checks sgl_decode_attention makes before it looks at its workspace
// (api.cu); sets *scale to the effective softmax scale.
sgl_status validate_decode_call(const void* q, const void* pool_k, const void* pool_v,
                                const int32_t* req_to_token, int32_t rtt_rows, int32_t rtt_stride,
                                const int32_t* req_pool_idx, const int32_t* seq_lens, int32_t batch,
                                int32_t max_seq_len, const void* out, const sgl_attn_dims* dims,
                                float* scale);

// The tensor-core pass of cascade decode: per (group, KV head, block of
// members) the members' decode queries attend to the group's keys and every
// row's fp32 softmax state goes to entry
// ((part_base + member * max_depth + depth) * Hkv + kvh) * G + head % G.
struct GroupArgs {
  const void* q;
  const void* pool_k;
  const void* pool_v;
  const int32_t* req_to_token;
  int32_t rtt_stride;
  const int32_t* req_pool_idx;
  const int32_t* group_start;
  const int32_t* group_len;
  const int32_t* group_depth;
  const int32_t* member_off;
  const int32_t* members;
  int32_t batch, n_groups, max_members, max_depth;
  void* part_ml;   // float2 entries
  void* part_acc;  // D floats per entry
  int64_t part_base;
  int* status;
  int32_t num_q_heads, num_kv_heads, head_dim;
  float sm_scale;
  // e4m3 pool: the K scale folds into the scores; the states' P.V rows stay
  // in code units
  bool kv_fp8 = false;
  float k_scale = 1.f;
};
// dependent: launched with programmatic stream serialization (it may start
// while the split kernel before it runs, and waits for it at its end)
sgl_status launch_cascade_groups(const GroupArgs& a, cudaStream_t stream, bool dependent = false);

// Whether kernel Kern was built with at least `regs` registers a thread (its
// launch allocation; read once).  A kernel that moves registers between its
// warpgroups with setmaxnreg needs exactly the launch registers it was split
// for: with fewer the increase would wait forever, so it is not launched.
template <auto Kern>
bool kernel_regs_at_least(int regs) {
  static std::atomic<int> cache{0};
  int r = cache.load(std::memory_order_relaxed);
  if (r == 0) {
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, Kern) != cudaSuccess) return false;
    r = fa.numRegs;
    cache.store(r, std::memory_order_relaxed);
  }
  return r >= regs;
}

// Launches kern<<<grid, block, smem, stream>>>(args...) with programmatic
// stream serialization: the kernel may start once every CTA of the kernel
// before it in the stream has signalled (grid_dep_launch) or exited, and
// must call grid_dep_wait before it reads what that kernel writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                             Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

struct ExtendArgs {
  const void* q;
  const void* k_new;
  const void* v_new;
  const void* pool_k;
  const void* pool_v;
  const int32_t* req_to_token;
  int32_t rtt_stride;
  const int32_t* req_pool_idx;
  const int32_t* prefix_lens;
  const int32_t* extend_lens;
  int32_t batch, total_extend, max_extend;
  int64_t pool_size;
  void* out;
  void* workspace;
  int32_t num_q_heads, num_kv_heads, head_dim;
  float sm_scale;
  // e4m3 pool (kv_fp8): every key and value, the suffix's included, is read
  // from the pool through req_to_token; k_new / v_new are unused
  bool kv_fp8 = false;
  float k_scale = 1.f, v_scale = 1.f;
};
size_t extend_workspace_bytes();
sgl_status launch_extend(const ExtendArgs& a, cudaStream_t stream);

// One launch for an extend batch and a plain decode batch over the same bf16
// pools (mixed.cu): persistent CTAs, one an SM, the first extend_ctas taking
// extend tiles first and the rest decode work first.  Shapes the single launch
// is not built for (mixed_launch_built false) run the two kernels in turn.
// Words 1..3 of the extend workspace hold the launch's work counters.
bool mixed_launch_built(const ExtendArgs& e, const DecodeArgs& d);
sgl_status launch_mixed(const ExtendArgs& e, const DecodeArgs& d, int32_t extend_ctas, cudaStream_t stream);

}  // namespace sgl
